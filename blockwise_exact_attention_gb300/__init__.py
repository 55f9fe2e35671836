"""Blockwise exact attention on GB300 (sm_103a).

Public API (all calls run in libbea.so's CUDA kernels on the current stream):

* ``flash_mha_fwd(q, k, v, softmax_scale, is_causal, window_size) -> (out, lse)``
* ``flash_mha_bwd(dout, q, k, v, out, lse, ...) -> (dq, dk, dv)``
* ``flash_mha_bwd_prepare / flash_mha_bwd_kv_block / flash_mha_bwd_finish``:
  the same backward in stages, dQ accumulated over several K/V blocks
* ``ring_merge(out_acc, lse_acc, out_blk, lse_blk, out_final=None)``
* ``flash_mha_fwd_merge(q, k, v, out_acc, lse_acc, ...)``: the fused ring
  step (a block's forward folded into the accumulator)
* ``ring_attention_fwd / ring_attention_bwd``: ring attention replayed as
  chunk steps on one GPU (``ring_attention_fwd_steps / ring_attention_bwd_steps``:
  the library's one-call form of the same replay).
* ``flash_attention / ring_attention``: the same as torch.autograd functions
  (the backward recomputed from the saved log-sum-exp).

The seeded input generators live in ``workloads`` and import nothing else.
"""
from .ops import (  # noqa: F401
    bwd_workspace_bytes,
    device_status,
    flash_mha_bwd,
    flash_mha_bwd_finish,
    flash_mha_bwd_kv_block,
    flash_mha_bwd_prepare,
    flash_mha_fwd,
    flash_mha_fwd_merge,
    launches_since_reset,
    ring_attention_bwd_steps,
    ring_attention_fwd_steps,
    ring_bwd_workspace_bytes,
    ring_merge,
    selftest_wait_timeout,
    selftest_inject_abort,
)
from .ring import chunk_schedule, ring_attention_bwd, ring_attention_fwd  # noqa: F401
from .autograd import flash_attention, ring_attention  # noqa: F401,E402
