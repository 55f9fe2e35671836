"""Ring attention over a sequence sharded across ranks (one GPU per rank).

flash_attn_jax flash_sharding.py, "Ring Forward" and "Ring Backward";
picotron context_parallel.py, RingAttentionFunc. Rank r of a ring of W ranks
holds query, key and value chunk r of the sequence. At ring step t it holds
the K/V chunk that started on rank (r - t) mod W (the pages' ppermute sends
r -> r + 1): it computes that block against its queries, with the key chunk
placed at its distance (j - r) c from the query chunk, and folds the block
into its running fp32 (out, lse) by the log-sum-exp merge. A block whose keys
are all masked (under a causal mask every chunk above the diagonal; under a
window every chunk beyond it) is skipped, while K/V keep moving.

The backward differentiates every live chunk pair once with the final out/lse
of the query rows. dQ of the local queries accumulates in the staged
backward's fp32 workspace; dK and dV accumulators travel around the ring with
their K/V chunk (picotron RingAttentionFunc.backward), each rank adding its
contribution before passing them on, so that after W steps every chunk's
gradients are back home carrying every rank's share. (flash_sharding.py's
ring_bwd instead rotates dout, q, out, lse and recomputes every pair twice;
the travelling accumulators compute each pair once.)

Exchange. torch.distributed point-to-point on the caller's process group:
each step sends this rank's current buffers to rank r + 1 and receives the
next ones from rank r - 1 into a second buffer. The K/V exchange of step t+1
is posted before step t's block is computed, so it overlaps the compute; the
travelling dK/dV leave after the block that adds to them. A rank's kernels
never wait on another rank's kernels: every exchange completes on the host
(the request is waited on) before its buffer is used. Backends that move
only host tensors (gloo) get device tensors staged through host copies.

The per-step compute goes through a step object; the default runs the
library's kernels (flash_mha_fwd / flash_mha_fwd_merge, the staged backward).
"""

from __future__ import annotations

import math

import torch
import torch.distributed as dist

from . import ops


def band_has_keys(c: int, is_causal: bool, window, key_offset: int) -> bool:
    """Whether any of c query rows sees any of c keys whose key 0 sits at query
    position key_offset: key j is visible to query r iff r - left <= j + key_offset
    <= r + right (an unbounded side is -1; causal forces right = 0)."""
    left, right = int(window[0]), int(window[1])
    if is_causal:
        right = 0
    lo = -(c - 1) if left < 0 else max(-left - key_offset, -(c - 1))
    hi = c - 1 if right < 0 else min(right - key_offset, c - 1)
    return lo <= hi


class CudaRingStep:
    """The per-step compute of the sharded ring on this rank's GPU (the library's kernels)."""

    def fwd_first(self, q, k, v, out_acc, lse, softmax_scale, is_causal, window):
        # the diagonal block (key offset 0) initialises the accumulator
        ops.flash_mha_fwd(q, k, v, softmax_scale, is_causal, window, out=out_acc, lse=lse)

    def fwd_merge(self, q, k, v, out_acc, lse, softmax_scale, is_causal, window, key_offset):
        ops.flash_mha_fwd_merge(q, k, v, out_acc, lse, softmax_scale, is_causal, window, key_offset=key_offset)

    def bwd_begin(self, dout, out, lse):
        self.ws = torch.empty(max(ops.bwd_workspace_bytes(dout), 256), dtype=torch.uint8, device=dout.device)
        ops.flash_mha_bwd_prepare(dout, out, lse, self.ws)

    def bwd_pair(self, dout, q, k, v, dk_acc, dv_acc, softmax_scale, is_causal, window, key_offset):
        ops.flash_mha_bwd_kv_block(dout, q, k, v, dk_acc, dv_acc, softmax_scale, is_causal, window,
                                   accumulate=True, workspace=self.ws, key_offset=key_offset)

    def bwd_end(self, dq, softmax_scale):
        ops.flash_mha_bwd_finish(dq, softmax_scale, accumulate=False, workspace=self.ws)
        self.ws = None


class _Exchange:
    """Send to rank r + 1, receive from rank r - 1 (ranks of `group`)."""

    def __init__(self, group):
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)
        self.host_only = dist.get_backend(group) == "gloo"

        def glob(gr):
            return gr if group is None else dist.get_global_rank(group, gr)
        self.to = glob((self.rank + 1) % self.world)
        self.frm = glob((self.rank - 1) % self.world)

    def post(self, send, recv):
        """Start sending `send` to the next rank and receiving `recv` from the previous
        one; returns a handle whose wait() completes both and fills `recv`."""
        stage = self.host_only and any(t.is_cuda for t in send)
        s_bufs = [t.detach().cpu() for t in send] if stage else [t.contiguous() for t in send]
        r_bufs = [torch.empty(t.shape, dtype=t.dtype) for t in recv] if stage else list(recv)
        p2p = [dist.P2POp(dist.isend, t, self.to, self.group) for t in s_bufs]
        p2p += [dist.P2POp(dist.irecv, t, self.frm, self.group) for t in r_bufs]
        reqs = dist.batch_isend_irecv(p2p)
        return _Pending(reqs, r_bufs, recv, stage)


class _Pending:
    def __init__(self, reqs, bufs, dst, staged):
        self.reqs, self.bufs, self.dst, self.staged = reqs, bufs, dst, staged

    def wait(self):
        for r in self.reqs:
            r.wait()
        if self.staged:
            for b, d in zip(self.bufs, self.dst):
                d.copy_(b)


def ring_attention_fwd_sharded(q, k, v, group=None, softmax_scale=None, is_causal=True, window_size=(-1, -1),
                               step=None):
    """This rank's share of ring attention: q, k, v are query/key/value chunk `rank`
    ([n, c, h, d], [n, c, h_kv, d]) of a sequence of world_size * c positions.
    Returns (out, lse): fp32 [n, c, h, d] and [n, h, c] for the local queries."""
    step = step or CudaRingStep()
    ex = _Exchange(group)
    n, c, h, d = q.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    window = tuple(int(x) for x in window_size)
    out = torch.empty((n, c, h, d), dtype=torch.float32, device=q.device)
    lse = torch.empty((n, h, c), dtype=torch.float32, device=q.device)
    cur_k, cur_v = k, v
    for t in range(ex.world):
        j = (ex.rank - t) % ex.world
        pending = None
        if t + 1 < ex.world:
            nxt_k, nxt_v = torch.empty_like(k), torch.empty_like(v)
            pending = ex.post([cur_k, cur_v], [nxt_k, nxt_v])
        key_offset = (j - ex.rank) * c
        if t == 0:
            step.fwd_first(q, cur_k, cur_v, out, lse, softmax_scale, is_causal, window)
        elif band_has_keys(c, is_causal, window, key_offset):
            step.fwd_merge(q, cur_k, cur_v, out, lse, softmax_scale, is_causal, window, key_offset)
        if pending is not None:
            pending.wait()
            cur_k, cur_v = nxt_k, nxt_v
    return out, lse


def ring_attention_bwd_sharded(dout, q, k, v, out, lse, group=None, softmax_scale=None, is_causal=True,
                               window_size=(-1, -1), step=None):
    """Backward of ring_attention_fwd_sharded for this rank's chunk, from the final
    (out, lse) of the local queries. Returns fp32 (dq, dk, dv) of the local chunk."""
    step = step or CudaRingStep()
    ex = _Exchange(group)
    n, c, h, d = q.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    window = tuple(int(x) for x in window_size)
    dq = torch.empty((n, c, h, d), dtype=torch.float32, device=q.device)
    cur_k, cur_v = k, v
    # the accumulators of the chunk this rank holds; at step 0 that is its own
    cur_dk = torch.zeros(k.shape, dtype=torch.float32, device=k.device)
    cur_dv = torch.zeros(v.shape, dtype=torch.float32, device=v.device)
    step.bwd_begin(dout, out, lse)
    for t in range(ex.world):
        j = (ex.rank - t) % ex.world
        kv_pending = None
        if t + 1 < ex.world:
            nxt_k, nxt_v = torch.empty_like(k), torch.empty_like(v)
            kv_pending = ex.post([cur_k, cur_v], [nxt_k, nxt_v])
        key_offset = (j - ex.rank) * c
        if band_has_keys(c, is_causal, window, key_offset):
            step.bwd_pair(dout, q, cur_k, cur_v, cur_dk, cur_dv, softmax_scale, is_causal, window, key_offset)
        if ex.world > 1:
            # this rank's share is in; the accumulators move on with their chunk (after the
            # last step they arrive back home)
            nxt_dk, nxt_dv = torch.empty_like(cur_dk), torch.empty_like(cur_dv)
            d_pending = ex.post([cur_dk, cur_dv], [nxt_dk, nxt_dv])
            d_pending.wait()
            cur_dk, cur_dv = nxt_dk, nxt_dv
        if kv_pending is not None:
            kv_pending.wait()
            cur_k, cur_v = nxt_k, nxt_v
    step.bwd_end(dq, softmax_scale)
    return dq, cur_dk, cur_dv
