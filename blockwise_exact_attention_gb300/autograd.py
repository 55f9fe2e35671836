"""torch.autograd wrappers over the C ABI: attention that trains.

``flash_attention(q, k, v, ...)`` returns ``out`` and, in the backward pass,
runs the library's backward recomputed from the saved log-sum-exp (picotron
context_parallel.py, ``RingAttentionFunc.forward/backward``, which save
``out`` and ``lse`` for the backward in the same way). ``ring_attention``
does the same over ring chunk steps replayed on one GPU (flash_attn_jax
flash_sharding.py, "Ring Forward" / "Ring Backward"). Grouped-query K/V heads
are read in place: query head i uses K/V head i / (h / h_kv), and the K/V
gradients come back with the K/V shapes, summed over each group inside the
kernels (no ``repeat_kv``).

Only marshalling lives here: every forward and backward step runs in the
library's CUDA kernels.
"""

from __future__ import annotations

import math

import torch

from . import ops, ring


def _grad_in(dout: torch.Tensor, like: torch.Tensor) -> torch.Tensor:
    # autograd may hand back an expanded or strided gradient; the kernels read a
    # dense, contiguous [n, l, h, d] tensor in the input dtype
    return dout.to(like.dtype).contiguous()


class _FlashAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, softmax_scale, is_causal, window_size):
        out, lse = ops.flash_mha_fwd(q, k, v, softmax_scale, is_causal, window_size)
        ctx.save_for_backward(q, k, v, out, lse)
        ctx.args = (softmax_scale, is_causal, window_size)
        ctx.mark_non_differentiable(lse)
        return out, lse

    @staticmethod
    def backward(ctx, dout, _dlse):
        q, k, v, out, lse = ctx.saved_tensors
        softmax_scale, is_causal, window_size = ctx.args
        dq, dk, dv = ops.flash_mha_bwd(_grad_in(dout, q), q, k, v, out, lse, softmax_scale, is_causal, window_size)
        return dq, dk, dv, None, None, None


class _RingAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, n_chunks, softmax_scale, is_causal):
        out, lse = ring.ring_attention_fwd(q, k, v, n_chunks, softmax_scale, is_causal)
        ctx.save_for_backward(q, k, v, out, lse)
        ctx.args = (n_chunks, softmax_scale, is_causal)
        ctx.mark_non_differentiable(lse)
        return out, lse

    @staticmethod
    def backward(ctx, dout, _dlse):
        q, k, v, out, lse = ctx.saved_tensors
        n_chunks, softmax_scale, is_causal = ctx.args
        dq, dk, dv = ring.ring_attention_bwd(_grad_in(dout, q), q, k, v, out, lse, n_chunks, softmax_scale,
                                             is_causal)
        return dq.to(q.dtype), dk.to(k.dtype), dv.to(v.dtype), None, None, None


def flash_attention(q, k, v, softmax_scale=None, is_causal=False, window_size=(-1, -1), return_lse=False):
    """Differentiable exact attention. q [n, l, h, d], k/v [n, lk, h_kv, d]
    (bf16 with d in {64, 128}, or fp32) -> out [n, l, h, d] (and lse [n, h, l])."""
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(q.shape[-1])
    out, lse = _FlashAttention.apply(q, k, v, float(softmax_scale), bool(is_causal), tuple(window_size))
    return (out, lse) if return_lse else out


def ring_attention(q, k, v, n_chunks: int, softmax_scale=None, is_causal=True, return_lse=False):
    """Differentiable ring attention over ``n_chunks`` sequence chunks,
    replayed on one GPU; the same results as ``flash_attention`` up to
    rounding order."""
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(q.shape[-1])
    out, lse = _RingAttention.apply(q, k, v, int(n_chunks), float(softmax_scale), bool(is_causal))
    return (out, lse) if return_lse else out
