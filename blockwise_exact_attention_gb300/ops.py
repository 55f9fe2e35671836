"""Python entry points over the C ABI: flash_mha_fwd, flash_mha_bwd, ring_merge.

Names and argument order follow the API the pages expose
(flash_attn_jax flash_sharding.py: ``fwd(q, k, v, softmax_scale, is_causal,
window_size) -> (out, lse)``, ``bwd(dout, q, k, v, out, lse, ...) -> (dq, dk,
dv)``; picotron context_parallel.py ``update_out_and_lse``). PyTorch only
supplies device memory and the current stream; a tensor that is not on a
CUDA device, or a missing library, raises.
"""

from __future__ import annotations

import math

import torch

from . import _lib

_DT = {torch.bfloat16: _lib.BEA_BF16, torch.float32: _lib.BEA_F32}

_launches = 0  # kernels launched through this module since the last reset


def launches_since_reset(reset: bool = False) -> int:
    global _launches
    n = _launches
    if reset:
        _launches = 0
    return n


def _count() -> None:
    global _launches
    _launches += _lib.load().bea_last_launch_count()


def _desc(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live on a CUDA device")
    if t.dtype not in _DT:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return _lib.describe(t.data_ptr(), _DT[t.dtype], t.shape, t.stride())


def _ref(d):
    import ctypes
    return None if d is None else ctypes.byref(d)


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def flash_mha_fwd(q, k, v, softmax_scale=None, is_causal=False, window_size=(-1, -1), out=None, lse=None,
                  out_dtype=None):
    """Exact attention forward. q [n,l,h,d], k/v [n,lk,h_kv,d] -> (out [n,l,h,d], lse [n,h,l] fp32)."""
    lib = _lib.load()
    n, lq, h, d = q.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype or q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((n, h, lq), dtype=torch.float32, device=q.device)
    dq_, dk_, dv_, do_, dl_ = (_desc(x) for x in (q, k, v, out, lse))
    rc = lib.bea_flash_mha_fwd(_ref(dq_), _ref(dk_), _ref(dv_), _ref(do_), _ref(dl_), float(softmax_scale),
                               int(bool(is_causal)), int(window_size[0]), int(window_size[1]), _stream())
    _lib.check(rc, "flash_mha_fwd")
    _count()
    return out, lse


def flash_mha_fwd_merge(q, k, v, out_acc, lse_acc, softmax_scale=None, is_causal=False, window_size=(-1, -1),
                        out_final=None, key_offset=None):
    """Fused ring step: the forward of (q, k, v) folded into the fp32
    accumulator (out_acc, lse_acc) in place by the log-sum-exp merge;
    ``out_final`` (bf16) also receives the merged rows. ``key_offset``: the
    position of key 0 relative to query 0 (default lq - lk)."""
    if key_offset is None:
        key_offset = q.shape[1] - k.shape[1]
    lib = _lib.load()
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(q.shape[3])
    ds = [_desc(x) for x in (q, k, v, out_acc, lse_acc, out_final)]
    rc = lib.bea_flash_mha_fwd_merge(*[_ref(x) for x in ds], float(softmax_scale), int(bool(is_causal)),
                                     int(window_size[0]), int(window_size[1]), int(key_offset), _stream())
    _lib.check(rc, "flash_mha_fwd_merge")
    _count()
    return out_acc, lse_acc


def bwd_workspace_bytes(q) -> int:
    n, lq, h, d = q.shape
    return int(_lib.load().bea_flash_mha_bwd_workspace_size(n, lq, h, d))


def flash_mha_bwd(dout, q, k, v, out, lse, softmax_scale=None, is_causal=False, window_size=(-1, -1), dq=None,
                  dk=None, dv=None, accumulate=False, workspace=None, grad_dtype=None):
    """Backward from the given out/lse -> (dq, dk, dv). With ``accumulate``
    the gradients are added to the given fp32 dq/dk/dv."""
    lib = _lib.load()
    d = q.shape[3]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    gdt = grad_dtype or q.dtype
    if dq is None:
        dq = torch.empty(q.shape, dtype=gdt, device=q.device)
    if dk is None:
        dk = torch.empty(k.shape, dtype=gdt, device=q.device)
    if dv is None:
        dv = torch.empty(v.shape, dtype=gdt, device=q.device)
    nbytes = bwd_workspace_bytes(q)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    ds = [_desc(x) for x in (dout, q, k, v, out, lse, dq, dk, dv)]
    rc = lib.bea_flash_mha_bwd(*[_ref(x) for x in ds], float(softmax_scale), int(bool(is_causal)),
                               int(window_size[0]), int(window_size[1]), int(bool(accumulate)),
                               workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream())
    _lib.check(rc, "flash_mha_bwd")
    _count()
    return dq, dk, dv


def _ws_args(workspace, q_like):
    if workspace is None:
        raise ValueError("the staged backward needs the caller's workspace (bwd_workspace_bytes)")
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def flash_mha_bwd_prepare(dout, out, lse, workspace):
    """Stage 1 of the staged backward: D, lse*log2(e) and a zeroed fp32 dQ
    accumulator in ``workspace`` (bf16 inputs)."""
    lib = _lib.load()
    ds = [_desc(x) for x in (dout, out, lse)]
    wp, wb = _ws_args(workspace, dout)
    rc = lib.bea_flash_mha_bwd_prepare(*[_ref(x) for x in ds], wp, wb, _stream())
    _lib.check(rc, "flash_mha_bwd_prepare")
    _count()


def flash_mha_bwd_kv_block(dout, q, k, v, dk, dv, softmax_scale=None, is_causal=False, window_size=(-1, -1),
                           accumulate=False, workspace=None, key_offset=None):
    """Stage 2: one K/V block's dK, dV (written or added) and its share of dQ
    (added into the workspace accumulator). ``key_offset``: the position of
    this block's key 0 relative to query 0 (default lq - lk)."""
    if key_offset is None:
        key_offset = q.shape[1] - k.shape[1]
    lib = _lib.load()
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(q.shape[3])
    ds = [_desc(x) for x in (dout, q, k, v, dk, dv)]
    wp, wb = _ws_args(workspace, q)
    rc = lib.bea_flash_mha_bwd_kv_block(*[_ref(x) for x in ds], float(softmax_scale), int(bool(is_causal)),
                                        int(window_size[0]), int(window_size[1]), int(key_offset),
                                        int(bool(accumulate)), wp, wb, _stream())
    _lib.check(rc, "flash_mha_bwd_kv_block")
    _count()
    return dk, dv


def flash_mha_bwd_finish(dq, softmax_scale, accumulate=False, workspace=None):
    """Stage 3: dq = softmax_scale * accumulator (written, or added to an fp32 dq)."""
    lib = _lib.load()
    wp, wb = _ws_args(workspace, dq)
    rc = lib.bea_flash_mha_bwd_finish(_ref(_desc(dq)), float(softmax_scale), int(bool(accumulate)), wp, wb,
                                      _stream())
    _lib.check(rc, "flash_mha_bwd_finish")
    _count()
    return dq


def flash_mha_bwd_noalloc(dout, q, k, v, out, lse, dq, dk, dv, softmax_scale=None, is_causal=False,
                          window_size=(-1, -1), accumulate=False):
    """flash_mha_bwd for callers that cannot allocate: the workspace is the
    library's own fixed device array, and dq/dk/dv must be given."""
    lib = _lib.load()
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(q.shape[3])
    ds = [_desc(x) for x in (dout, q, k, v, out, lse, dq, dk, dv)]
    rc = lib.bea_flash_mha_bwd_noalloc(*[_ref(x) for x in ds], float(softmax_scale), int(bool(is_causal)),
                                       int(window_size[0]), int(window_size[1]), int(bool(accumulate)), _stream())
    _lib.check(rc, "flash_mha_bwd_noalloc")
    _count()
    return dq, dk, dv


def ring_merge(out_acc, lse_acc, out_blk, lse_blk, out_final=None):
    """Fold (out_blk, lse_blk) into the fp32 accumulator (out_acc, lse_acc) in place."""
    lib = _lib.load()
    ds = [_desc(x) for x in (out_acc, lse_acc, out_blk, lse_blk, out_final)]
    rc = lib.bea_ring_merge(*[_ref(x) for x in ds], _stream())
    _lib.check(rc, "ring_merge")
    _count()
    return out_acc, lse_acc


def ring_attention_fwd_steps(q, k, v, out_acc, lse, n_chunks, softmax_scale=None, is_causal=False,
                            window_size=(-1, -1), out_final=None):
    """The whole ring forward replay in one library call: every live chunk pair folded
    into the fp32 accumulator ``out_acc`` (and ``lse``), one launch per ring step;
    ``out_final`` (bf16) also receives the result."""
    lib = _lib.load()
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(q.shape[3])
    ds = [_desc(x) for x in (q, k, v, out_acc, lse, out_final)]
    rc = lib.bea_ring_attention_fwd(*[_ref(x) for x in ds], int(n_chunks), float(softmax_scale),
                                    int(bool(is_causal)), int(window_size[0]), int(window_size[1]), _stream())
    _lib.check(rc, "ring_attention_fwd")
    _count()
    return out_acc, lse


def ring_bwd_workspace_bytes(q, n_chunks) -> int:
    n, l, h, d = q.shape
    return int(_lib.load().bea_ring_attention_bwd_workspace_size(n, l, h, d, int(n_chunks)))


def ring_attention_bwd_steps(dout, q, k, v, out, lse, dq, dk, dv, n_chunks, softmax_scale=None, is_causal=False,
                            window_size=(-1, -1), workspace=None):
    """The whole ring backward replay in one library call: fp32 dq, dk, dv written."""
    lib = _lib.load()
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(q.shape[3])
    if workspace is None:
        workspace = torch.empty(max(ring_bwd_workspace_bytes(q, n_chunks), 256), dtype=torch.uint8, device=q.device)
    ds = [_desc(x) for x in (dout, q, k, v, out, lse, dq, dk, dv)]
    rc = lib.bea_ring_attention_bwd(*[_ref(x) for x in ds], int(n_chunks), float(softmax_scale),
                                    int(bool(is_causal)), int(window_size[0]), int(window_size[1]),
                                    workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream())
    _lib.check(rc, "ring_attention_bwd")
    _count()
    return dq, dk, dv


def device_status() -> int:
    """Synchronise, read and clear the device status word (0 = ok)."""
    return _lib.load().bea_get_device_status(_stream())


def selftest_wait_timeout(limit_us: int) -> None:
    _lib.check(_lib.load().bea_selftest_wait_timeout(int(limit_us), _stream()), "selftest_wait_timeout")


def selftest_inject_abort(tile: int) -> None:
    """Arm a one-shot abort of the next forward/backward main-kernel launch at
    tile `tile` of its first CTA (-1 disarms); see bea_selftest_inject_abort."""
    _lib.check(_lib.load().bea_selftest_inject_abort(int(tile)), "selftest_inject_abort")
