"""Ring attention replayed on one GPU as sequential chunk steps.

The sequence is split into ``n_chunks`` equal chunks. In ring attention the
device owning query chunk i holds, at step t, the K/V chunk that started on
device i - t (ppermute sends i -> i+1). With causal masking the step's chunk
pair is skipped when j > i, computed with the causal kernel on the diagonal
j == i and with the full kernel otherwise; every computed block is folded into
a running fp32 (out, lse) by the log-sum-exp merge (flash_attn_jax
flash_sharding.py, sections "Ring Forward" and "Ring Backward").

On one GPU the K/V "rotation" is a zero-copy chunk view of the resident
tensors, so the schedule reduces to a sequence of forward calls and merges,
all through the C ABI. The backward runs every visible chunk pair once with
the final out/lse of its query rows and adds the partial gradients in fp32;
for bf16 inputs it uses the staged backward, so that D is computed once per
query chunk and dQ stays in the fp32 workspace accumulator across its K/V
chunks.
"""

from __future__ import annotations

import math

import numpy as np
import torch

from . import ops


def chunk_schedule(n_chunks: int, is_causal: bool):
    """Per query chunk i: the ring steps [(t, j, kind)], kind in skip/causal/full."""
    sched = []
    for i in range(n_chunks):
        steps = []
        for t in range(n_chunks):
            j = (i - t) % n_chunks
            if not is_causal:
                kind = "full"
            elif j > i:
                kind = "skip"
            elif j == i:
                kind = "causal"
            else:
                kind = "full"
            steps.append((t, j, kind))
        sched.append(steps)
    return sched


def _chunks(x, n_chunks, dim):
    c = x.shape[dim] // n_chunks
    return [x.narrow(dim, i * c, c) for i in range(n_chunks)]


def _step_view(x, first: int, count: int, c: int, l_dim: int):
    """Chunks first .. first + count - 1 of a batch-1 sequence tensor as one batch of
    ``count`` chunks: [1, l, h, d] -> [count, c, h, d] (l_dim 1) or [1, h, l] ->
    [count, h, c] (l_dim 2). A zero-copy strided view: the batch stride is one chunk."""
    st = list(x.stride())
    size = list(x.shape)
    size[0], size[l_dim] = count, c
    st[0] = c * x.stride(l_dim)
    return x.as_strided(size, st, x.storage_offset() + first * c * x.stride(l_dim))


def _band_has_keys(c: int, is_causal: bool, window, key_offset: int) -> bool:
    """Whether any of c query rows sees any of c keys whose key 0 sits at query
    position key_offset (the window compares positions)."""
    left, right = int(window[0]), int(window[1])
    if is_causal:
        right = 0
    r = np.arange(c, dtype=np.int64)
    lo = np.zeros(c, dtype=np.int64) if left < 0 else np.maximum(r - left - key_offset, 0)
    hi = np.full(c, c - 1, dtype=np.int64) if right < 0 else np.minimum(r + right - key_offset, c - 1)
    return bool((lo <= hi).any())


def _ring_step_groups(n_chunks: int, is_causal: bool, cast: bool, window=(-1, -1), c: int = 1):
    """Per ring step t, the calls that cover its live chunk pairs: (first query chunk,
    first K/V chunk, number of consecutive chunks, key offset, whether this is those query
    chunks' last live step). Step t pairs query chunk i with K/V chunk (i - t) mod C: the
    pairs with i >= t share the key offset -t*c, the wrapped ones (i < t) (C - t)*c. A run
    of pairs whose key band is empty is skipped (under a causal mask: every wrapped pair;
    under a window: the pairs beyond it). When the result is cast at each query chunk's
    last live step, a run is split where that step changes."""
    C = n_chunks
    runs = []  # (t, i0, j0, cnt, koff)
    for t in range(C):
        for (i0, j0, cnt, koff) in ((t, 0, C - t, -t * c), (0, C - t, t, (C - t) * c)):
            if cnt > 0 and _band_has_keys(c, is_causal, window, koff):
                runs.append((t, i0, j0, cnt, koff))
    last = {}
    for (t, i0, _j0, cnt, _k) in runs:
        for i in range(i0, i0 + cnt):
            last[i] = max(last.get(i, -1), t)
    groups = [[] for _ in range(C)]
    for (t, i0, j0, cnt, koff) in runs:
        if not cast:
            groups[t].append((i0, j0, cnt, koff, False))
            continue
        u = 0
        while u < cnt:
            fin = last[i0 + u] == t
            v = u
            while v < cnt and (last[i0 + v] == t) == fin:
                v += 1
            groups[t].append((i0 + u, j0 + u, v - u, koff, fin))
            u = v
    return groups


def ring_attention_fwd(q, k, v, n_chunks: int, softmax_scale=None, is_causal=True, out_dtype=None,
                       block_dtype=None, fused=None, window_size=(-1, -1)):
    """Forward over ring chunk steps -> (out, lse).

    ``out_dtype`` fp32 makes the fp32 accumulator itself the result;
    otherwise (default: q's dtype) the last merge of each query chunk also
    writes the cast result. ``block_dtype`` is the dtype of each block's
    partial output (default: q's dtype, as the pages feed the kernel's
    q-dtype output into the fp32 merge). ``fused`` (default: on for bf16
    inputs when no block dtype is asked for) folds each block into the
    accumulator inside the forward kernel instead of writing it out and
    running ring_merge; the library then drives every ring step in one call
    (bea_ring_attention_fwd): one launch per ring step, consecutive launches
    chained by programmatic dependent launch. The unfused form composes the
    forward and ring_merge calls here, a pair of launches per ring step.

    Every query chunk steps through its K/V chunks in ring order. On one GPU
    the query chunks are independent, so all chunk pairs of one ring step run
    as one call over a batch of chunk views (ring step t pairs query chunk i
    with K/V chunk i - t). Batches larger than 1 run their rows one after
    another.
    ``window_size`` (fused steps only) masks every chunk pair by sequence
    position, with its key chunk placed at its distance from the query chunk;
    pairs entirely outside the window are skipped.
    """
    n, l, h, d = q.shape
    if l % n_chunks:
        raise ValueError("sequence length must split evenly into chunks")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    if fused is None:
        fused = q.dtype == torch.bfloat16 and block_dtype is None
    window_size = tuple(int(x) for x in window_size)
    if window_size != (-1, -1) and not fused:
        raise ValueError("a windowed ring runs as fused ring steps (bf16 inputs, no block dtype)")
    out_dtype = out_dtype or q.dtype
    block_dtype = block_dtype or q.dtype
    dev = q.device
    out = torch.empty(q.shape, dtype=out_dtype, device=dev)
    lse = torch.empty((n, h, l), dtype=torch.float32, device=dev)
    acc = out if out_dtype == torch.float32 else torch.empty(q.shape, dtype=torch.float32, device=dev)
    c = l // n_chunks
    cast = out_dtype != torch.float32
    if fused:
        # the library drives every ring step itself: one launch per step, chained on the stream
        ops.ring_attention_fwd_steps(q, k, v, acc, lse, n_chunks, softmax_scale, is_causal, window_size,
                                     out_final=out if cast else None)
        return out, lse
    for b in range(n):
        qb, kb, vb = q[b:b + 1], k[b:b + 1], v[b:b + 1]
        accb, outb, lseb = acc[b:b + 1], out[b:b + 1], lse[b:b + 1]
        for t, parts in enumerate(_ring_step_groups(n_chunks, is_causal, cast, window_size, c)):
            for (i0, j0, cnt, koff, final) in parts:
                qv, kv_, vv = (_step_view(x_, f, cnt, c, 1) for x_, f in ((qb, i0), (kb, j0), (vb, j0)))
                av, lv = _step_view(accb, i0, cnt, c, 1), _step_view(lseb, i0, cnt, c, 2)
                fin = _step_view(outb, i0, cnt, c, 1) if (final and cast) else None
                if t == 0:
                    # the first block (the diagonal, key offset 0) initialises the accumulator
                    # (merge with (0, -inf) is the identity); a chunk whose only block this is
                    # gets its final output at once
                    ops.flash_mha_fwd(qv, kv_, vv, softmax_scale, is_causal, window_size,
                                      out=fin if fin is not None else av, lse=lv)
                else:
                    causal = False  # no window: a live off-diagonal pair sees all its keys
                    blk = torch.empty((cnt, c, h, d), dtype=block_dtype, device=dev)
                    lblk = torch.empty((cnt, h, c), dtype=torch.float32, device=dev)
                    ops.flash_mha_fwd(qv, kv_, vv, softmax_scale, causal, out=blk, lse=lblk)
                    ops.ring_merge(av, lv, blk, lblk, out_final=fin)
    return out, lse


def ring_attention_bwd(dout, q, k, v, out, lse, n_chunks: int, softmax_scale=None, is_causal=True,
                       window_size=(-1, -1)):
    """Backward over every live chunk pair -> fp32 (dq, dk, dv).

    ``window_size`` masks each chunk pair by sequence position (key chunk
    placed at its distance from the query chunk, bf16 inputs only); pairs
    with no visible key are skipped. bf16 inputs run in one library call
    (bea_ring_attention_bwd: all chunk pairs of a ring step in one launch);
    fp32 inputs compose one backward call per chunk pair here.
    """
    n, l, h, d = q.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    window_size = tuple(int(x) for x in window_size)
    dev = q.device
    dq = torch.empty(q.shape, dtype=torch.float32, device=dev)
    dk = torch.empty(k.shape, dtype=torch.float32, device=dev)
    dv = torch.empty(v.shape, dtype=torch.float32, device=dev)
    if q.dtype == torch.bfloat16:
        # the library drives every ring step itself: one preprocess, one launch per ring
        # step (all its chunk pairs), one dQ conversion
        return ops.ring_attention_bwd_steps(dout, q, k, v, out, lse, dq, dk, dv, n_chunks, softmax_scale, is_causal,
                                            window_size)
    if not is_causal:
        dq.zero_()
        dk.zero_()
        dv.zero_()
    ws = torch.empty(ops.bwd_workspace_bytes(_chunks(q, n_chunks, 1)[0]), dtype=torch.uint8, device=dev)
    qs, ks, vs = _chunks(q, n_chunks, 1), _chunks(k, n_chunks, 1), _chunks(v, n_chunks, 1)
    dos, os_, ls = _chunks(dout, n_chunks, 1), _chunks(out, n_chunks, 1), _chunks(lse, n_chunks, 2)
    dqs, dks, dvs = _chunks(dq, n_chunks, 1), _chunks(dk, n_chunks, 1), _chunks(dv, n_chunks, 1)
    c = l // n_chunks
    staged = q.dtype == torch.bfloat16
    if window_size != (-1, -1) and not staged:
        raise ValueError("a windowed ring backward needs bf16 inputs")
    for i in range(n_chunks):
        live = []
        for t in range(n_chunks):
            j = (i - t) % n_chunks
            if _band_has_keys(c, is_causal, window_size, (j - i) * c):
                live.append(j)
        if staged:
            # D of query chunk i once, its dQ summed over every visible K/V chunk in the fp32
            # workspace accumulator, one conversion at the end
            ops.flash_mha_bwd_prepare(dos[i], os_[i], ls[i], ws)
        for j in live:
            # causal, query chunks in ascending order: the diagonal pair (i, i) is the
            # first to touch dk_i and dv_i, so it overwrites instead of adding
            first = is_causal and j == i
            if staged:
                ops.flash_mha_bwd_kv_block(dos[i], qs[i], ks[j], vs[j], dks[j], dvs[j], softmax_scale,
                                           is_causal, window_size, accumulate=not first, workspace=ws,
                                           key_offset=(j - i) * c)
            else:
                ops.flash_mha_bwd(dos[i], qs[i], ks[j], vs[j], os_[i], ls[i], softmax_scale, is_causal and j == i,
                                  dq=dqs[i], dk=dks[j], dv=dvs[j], accumulate=not first, workspace=ws)
        if staged:
            # the diagonal pair (key offset 0) always has visible keys, so `live` is never empty
            ops.flash_mha_bwd_finish(dqs[i], softmax_scale, accumulate=False, workspace=ws)
    return dq, dk, dv
