"""Plain fp64 CPU oracle for blockwise exact attention.

TEST INFRASTRUCTURE. This module is the independent definition that the CUDA
path is checked against. Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it; the
product path never does, and this module imports nothing from the product
package.

What it computes is the plain definition of exact softmax attention. The
blockwise/online-softmax method reaches the same numbers up to rounding order,
so no step of the blocked algorithm is replayed here:

* forward: picotron ``parallel/context_parallel.py``, function
  ``ring_attention_forward`` (scores, causal mask, softmax, log-sum-exp, P V);
* backward recomputed from the log-sum-exp: the same page, function
  ``ring_attention_backward`` (Steps 1-6: dV, dP, D, dS, dQ, dK);
* grouped-query head mapping: the same page, ``RingAttention._repeat_kv``
  (query head i reads K/V head i // (h / h_kv));
* the ``[n, h, l]`` log-sum-exp layout, the fp32/fp64 running accumulator
  initialised to (0, -inf) and the max/log1p merge: flash_attn_jax
  ``flash_sharding.py``, section "Ring Forward" (``ring_fwd``);
* the sigmoid form of the merge: picotron ``update_out_and_lse``;
* the causal chunk schedule of the ring (skip / causal / full by comparing the
  K/V chunk index with the query chunk index, K/V moving i -> i+1 each step):
  ``flash_sharding.py`` "Ring Forward" and "Ring Backward".

Readings taken where the pages are silent:

* window ``(left, right)``: key j is visible to query i iff
  ``(left < 0 or j >= i - left) and (right < 0 or j <= i + right)``;
  ``is_causal`` means ``right = 0``.
* key positions: key j sits at position ``j + key_offset`` of the query
  positions, and the window compares positions:
  ``(left < 0 or j + key_offset >= i - left) and (right < 0 or j + key_offset <= i + right)``.
  By default ``key_offset = lq - lk``: with ``lq != lk`` the last query row is
  aligned with the last key (bottom-right alignment; the pages only use
  ``lq == lk``, where the offset is 0). Ring chunk pairs pass the distance
  between their key chunk and their query chunk.
* a query row with no visible key has ``out = 0``, ``lse = -inf`` and zero
  gradients (the skipped-block convention of ``ring_fwd``, applied per row).
* merging two rows that both have ``lse = -inf`` leaves the accumulator as it
  is; when exactly one side is ``-inf`` the other side is taken exactly.

Every function works in float64 on whatever array it is given (bf16 inputs are
passed in already upcast, so the oracle sees exactly the uploaded bits).
"""

from __future__ import annotations

import math

import numpy as np

NEG_INF = float("-inf")

__all__ = [
    "visible_mask",
    "attention_fwd",
    "attention_probs",
    "attention_bwd",
    "merge_max_form",
    "merge_sigmoid_form",
    "ring_chunk_schedule",
    "ring_fwd_replay",
    "ring_bwd_replay",
    "algorithmic_flops",
    "visible_pairs",
]


# ---------------------------------------------------------------------------
# masks
# ---------------------------------------------------------------------------

def _effective_window(is_causal: bool, window: tuple[int, int]) -> tuple[int, int]:
    left, right = int(window[0]), int(window[1])
    if is_causal:
        if right > 0:
            raise ValueError("is_causal with window right > 0 is contradictory")
        right = 0
    return left, right


def visible_mask(rows: np.ndarray, lk: int, is_causal: bool,
                 window: tuple[int, int] = (-1, -1), key_offset: int = 0) -> np.ndarray:
    """Boolean ``[len(rows), lk]``: True where query ``rows[r]`` may see key ``j``.

    Causal masking as in picotron ``ring_attention_forward`` (entries above the
    diagonal are masked); the window and the key offset are the readings stated
    in the module doc.
    """
    left, right = _effective_window(is_causal, window)
    i = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.arange(lk, dtype=np.int64)[None, :] + int(key_offset)
    vis = np.ones((i.shape[0], lk), dtype=bool)
    if left >= 0:
        vis &= j >= i - left
    if right >= 0:
        vis &= j <= i + right
    return vis


def _key_band(r0: int, r1: int, lk: int, is_causal: bool,
              window: tuple[int, int], key_offset: int = 0) -> tuple[int, int]:
    """Keys that any of the query rows ``[r0, r1)`` can see (all others are
    masked, so dropping them changes no sum)."""
    left, right = _effective_window(is_causal, window)
    k0 = 0 if left < 0 else min(lk, max(0, r0 - left - key_offset))
    k1 = lk if right < 0 else max(0, min(lk, r1 - 1 + right - key_offset + 1))
    return k0, max(k0, k1)


def _key_offset(lq: int, lk: int, key_offset) -> int:
    """The default key offset: bottom-right alignment (0 when lq == lk)."""
    return lq - lk if key_offset is None else int(key_offset)


def _check_shapes(q, k, v, is_causal, window):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [n, l, h, d]")
    n, lq, h, d = q.shape
    nk, lk, hkv, dk = k.shape
    if (nk, dk) != (n, d) or v.shape != k.shape:
        raise ValueError("k, v must be [n, lk, h_kv, d] matching q")
    if hkv == 0 or h % hkv != 0:
        raise ValueError("h must be a multiple of h_kv")
    _effective_window(is_causal, window)
    return n, lq, lk, h, hkv, d


# ---------------------------------------------------------------------------
# forward
# ---------------------------------------------------------------------------

def attention_fwd(q, k, v, softmax_scale: float, is_causal: bool = False,
                  window: tuple[int, int] = (-1, -1), rows=None,
                  row_block: int = 1024, key_offset=None):
    """Exact attention forward in fp64: returns ``(out [n,l,h,d], lse [n,h,l])``.

    For each batch b and query head hq (K/V head ``hq // g``):
    ``S = softmax_scale * Q K^T``, masked entries set to -inf,
    ``lse_i = log sum_j exp(S_ij)`` (natural log, scale included),
    ``P = exp(S - lse)``, ``out = P V``.

    ``rows`` (optional) restricts the computation to those absolute query row
    indices; the result then has ``len(rows)`` rows in place of ``lq``.
    ``key_offset`` places key j at query position ``j + key_offset`` (default:
    ``lq - lk``, bottom-right alignment).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, lq, lk, h, hkv, d = _check_shapes(q, k, v, is_causal, window)
    off = _key_offset(lq, lk, key_offset)
    g = h // hkv
    if rows is None:
        rows = np.arange(lq, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    nr = rows.shape[0]
    out = np.zeros((n, nr, h, d), dtype=np.float64)
    lse = np.full((n, h, nr), NEG_INF, dtype=np.float64)
    for r0 in range(0, nr, row_block):
        r1 = min(nr, r0 + row_block)
        idx = rows[r0:r1]
        k0, k1 = _key_band(int(idx.min()), int(idx.max()) + 1, lk, is_causal, window, off)
        if k1 <= k0:
            continue
        vis = visible_mask(idx, lk, is_causal, window, off)[:, k0:k1]
        any_vis = vis.any(axis=1)
        for b in range(n):
            for hq in range(h):
                kv = hq // g
                s = softmax_scale * (q[b, idx, hq, :] @ k[b, k0:k1, kv, :].T)
                s = np.where(vis, s, NEG_INF)
                m = np.where(any_vis, s.max(axis=1, initial=NEG_INF), 0.0)
                e = np.exp(s - m[:, None])            # masked -> exp(-inf) = 0
                ssum = e.sum(axis=1)
                with np.errstate(divide="ignore"):
                    row_lse = np.where(any_vis, m + np.log(ssum), NEG_INF)
                p = np.where(any_vis[:, None], e / np.where(any_vis, ssum, 1.0)[:, None], 0.0)
                out[b, r0:r1, hq, :] = p @ v[b, k0:k1, kv, :]
                lse[b, hq, r0:r1] = row_lse
    return out, lse


def attention_probs(q, k, softmax_scale: float, is_causal: bool = False,
                    window: tuple[int, int] = (-1, -1), key_offset=None):
    """The full probability matrix ``P [n, h, lq, lk]`` (small inputs only)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    n, lq, h, d = q.shape
    lk, hkv = k.shape[1], k.shape[2]
    g = h // hkv
    vis = visible_mask(np.arange(lq), lk, is_causal, window, _key_offset(lq, lk, key_offset))
    any_vis = vis.any(axis=1)
    P = np.zeros((n, h, lq, lk))
    for b in range(n):
        for hq in range(h):
            s = softmax_scale * (q[b, :, hq, :] @ k[b, :, hq // g, :].T)
            s = np.where(vis, s, NEG_INF)
            m = np.where(any_vis, s.max(axis=1, initial=NEG_INF), 0.0)
            e = np.exp(s - m[:, None])
            tot = np.where(any_vis, e.sum(axis=1), 1.0)
            P[b, hq] = np.where(any_vis[:, None], e / tot[:, None], 0.0)
    return P


# ---------------------------------------------------------------------------
# backward (recomputed from lse)
# ---------------------------------------------------------------------------

def attention_bwd(dout, q, k, v, out, lse, softmax_scale: float,
                  is_causal: bool = False, window: tuple[int, int] = (-1, -1),
                  row_block: int = 1024, key_offset=None):
    """Analytic backward in fp64 from the GIVEN ``out`` and ``lse``.

    ``P = exp(S - lse)`` (masked entries 0), ``dV = P^T dO``, ``dP = dO V^T``,
    ``D = rowsum(dO * out)``, ``dS = P * (dP - D)``, ``dQ = scale * dS K``,
    ``dK = scale * dS^T Q``; dK and dV of a K/V head are summed over the query
    heads that read it. Using the given out/lse (not recomputed ones) is what
    makes per-chunk gradients of the ring add up exactly (flash_sharding.py,
    "Ring Backward": every chunk pair uses the final out/lse of its rows).
    Rows whose lse is -inf contribute nothing.
    """
    dout = np.asarray(dout, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    out = np.asarray(out, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    n, lq, lk, h, hkv, d = _check_shapes(q, k, v, is_causal, window)
    off = _key_offset(lq, lk, key_offset)
    g = h // hkv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for r0 in range(0, lq, row_block):
        r1 = min(lq, r0 + row_block)
        idx = np.arange(r0, r1)
        k0, k1 = _key_band(r0, r1, lk, is_causal, window, off)
        if k1 <= k0:
            continue
        vis = visible_mask(idx, lk, is_causal, window, off)[:, k0:k1]
        for b in range(n):
            for hq in range(h):
                kv = hq // g
                L = lse[b, hq, r0:r1]
                live = np.isfinite(L)
                s = softmax_scale * (q[b, r0:r1, hq, :] @ k[b, k0:k1, kv, :].T)
                p = np.where(vis & live[:, None],
                             np.exp(s - np.where(live, L, 0.0)[:, None]), 0.0)
                do = dout[b, r0:r1, hq, :]
                dv[b, k0:k1, kv, :] += p.T @ do                     # Step 1
                dp = do @ v[b, k0:k1, kv, :].T                      # Step 2
                D = np.sum(do * out[b, r0:r1, hq, :], axis=1)       # Step 3
                ds = p * (dp - D[:, None])                          # Step 4
                ds = np.where(vis, ds, 0.0)
                dq[b, r0:r1, hq, :] = softmax_scale * (ds @ k[b, k0:k1, kv, :])   # Step 5
                dk[b, k0:k1, kv, :] += softmax_scale * (ds.T @ q[b, r0:r1, hq, :])  # Step 6
    return dq, dk, dv


# ---------------------------------------------------------------------------
# merge of partial (out, lse) pairs
# ---------------------------------------------------------------------------

def _rows_view(lse):
    """lse [n, h, l] -> broadcastable [n, l, h, 1] against out [n, l, h, d]."""
    return np.transpose(lse, (0, 2, 1))[..., None]


def merge_max_form(out_a, lse_a, out_b, lse_b):
    """Fold block ``(out_b, lse_b)`` into the running ``(out_a, lse_a)``.

    flash_sharding.py "Ring Forward": ``mx = max(la, lb)``, ``mn = min(la, lb)``,
    ``l = log1p(exp(mn - mx)) + mx``, ``o = oa*exp(la - l) + ob*exp(lb - l)``.
    Guards (reading): both -inf -> the running pair is kept; one side -inf ->
    the other side exactly.
    """
    out_a = np.asarray(out_a, dtype=np.float64)
    out_b = np.asarray(out_b, dtype=np.float64)
    la = np.asarray(lse_a, dtype=np.float64)
    lb = np.asarray(lse_b, dtype=np.float64)
    mx = np.maximum(la, lb)
    mn = np.minimum(la, lb)
    both_dead = np.isneginf(mx)
    safe_mx = np.where(both_dead, 0.0, mx)
    with np.errstate(invalid="ignore"):
        l_new = np.where(both_dead, NEG_INF, np.log1p(np.exp(mn - safe_mx)) + safe_mx)
    safe_l = np.where(both_dead, 0.0, l_new)
    wa = np.where(both_dead, 1.0, np.exp(la - safe_l))
    wb = np.where(both_dead, 0.0, np.exp(lb - safe_l))
    o = out_a * _rows_view(wa) + out_b * _rows_view(wb)
    return o, l_new


def merge_sigmoid_form(out_a, lse_a, out_b, lse_b):
    """The same fold in picotron's form (``update_out_and_lse``):
    ``o <- o - sigmoid(lb - la) * (o - ob)``, ``l <- l - logsigmoid(la - lb)``.
    Guards as in :func:`merge_max_form`.
    """
    out_a = np.asarray(out_a, dtype=np.float64)
    out_b = np.asarray(out_b, dtype=np.float64)
    la = np.asarray(lse_a, dtype=np.float64)
    lb = np.asarray(lse_b, dtype=np.float64)
    a_dead = np.isneginf(la)
    b_dead = np.isneginf(lb)
    live = ~(a_dead | b_dead)
    with np.errstate(invalid="ignore"):
        x = np.where(live, lb - la, 0.0)      # sigmoid argument
    sig = np.where(x >= 0, 1.0 / (1.0 + np.exp(-np.abs(x))),
                   np.exp(-np.abs(x)) / (1.0 + np.exp(-np.abs(x))))
    # -logsigmoid(la - lb) = softplus(lb - la) = max(x, 0) + log1p(exp(-|x|))
    softplus = np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))
    w = np.where(live, sig, np.where(a_dead & ~b_dead, 1.0, 0.0))
    o = out_a - _rows_view(w) * (out_a - out_b)
    l_new = np.where(live, la + softplus, np.where(a_dead, lb, la))
    return o, l_new


# ---------------------------------------------------------------------------
# ring replay (one process; the K/V rotation becomes a chunk index)
# ---------------------------------------------------------------------------

def ring_chunk_schedule(n_chunks: int, is_causal: bool):
    """Per query chunk i: the list of (step t, kv chunk j, kind) in ring order.

    The K/V chunk held at step t by the device that owns query chunk i came
    from device i - t (ppermute sends i -> i+1), so ``j = (i - t) mod N``.
    kind is ``"skip"`` when j > i under causal masking, ``"causal"`` on the
    diagonal j == i, ``"full"`` otherwise (flash_sharding.py, "Ring Forward").
    """
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


def ring_fwd_replay(q, k, v, softmax_scale: float, n_chunks: int, is_causal: bool,
                    window: tuple[int, int] = (-1, -1)):
    """Forward of ring attention on sequence chunks, folded with the merge.

    Each query chunk starts from the accumulator (0, -inf) and folds in the
    block result of every K/V chunk in ring order; skipped chunks contribute
    (0, -inf). With a window, every chunk pair is masked by positions (its key
    chunk placed at offset ``(j - i) * c`` from its query chunk).
    """
    q = np.asarray(q, dtype=np.float64)
    n, l, h, d = q.shape
    if l % n_chunks:
        raise ValueError("sequence must split evenly into chunks")
    c = l // n_chunks
    out = np.zeros_like(q)
    lse = np.full((n, h, l), NEG_INF)
    for i, steps in enumerate(ring_chunk_schedule(n_chunks, is_causal)):
        qs = slice(i * c, (i + 1) * c)
        o_acc = np.zeros((n, c, h, d))
        l_acc = np.full((n, h, c), NEG_INF)
        for _t, j, kind in steps:
            ks = slice(j * c, (j + 1) * c)
            if tuple(window) != (-1, -1):
                o_b, l_b = attention_fwd(q[:, qs], k[:, ks], v[:, ks], softmax_scale, is_causal, window,
                                         key_offset=(j - i) * c)
            elif kind == "skip":
                continue
            else:
                o_b, l_b = attention_fwd(q[:, qs], k[:, ks], v[:, ks], softmax_scale,
                                         is_causal=(kind == "causal"))
            o_acc, l_acc = merge_max_form(o_acc, l_acc, o_b, l_b)
        out[:, qs] = o_acc
        lse[:, :, qs] = l_acc
    return out, lse


def ring_bwd_replay(dout, q, k, v, out, lse, softmax_scale: float, n_chunks: int,
                    is_causal: bool, window: tuple[int, int] = (-1, -1)):
    """Backward of ring attention: every visible chunk pair (i, j) runs the
    block backward with the FINAL out/lse of query chunk i, and the partial
    gradients are summed (flash_sharding.py, "Ring Backward"). One process
    computes each pair once."""
    q = np.asarray(q, dtype=np.float64)
    n, l, h, d = q.shape
    c = l // n_chunks
    dq = np.zeros_like(q)
    dk = np.zeros(np.shape(k))
    dv = np.zeros(np.shape(v))
    for i, steps in enumerate(ring_chunk_schedule(n_chunks, is_causal)):
        qs = slice(i * c, (i + 1) * c)
        for _t, j, kind in steps:
            ks = slice(j * c, (j + 1) * c)
            if tuple(window) != (-1, -1):
                a, b_, c_ = attention_bwd(dout[:, qs], q[:, qs], k[:, ks], v[:, ks],
                                          out[:, qs], lse[:, :, qs], softmax_scale,
                                          is_causal, window, key_offset=(j - i) * c)
            elif kind == "skip":
                continue
            else:
                a, b_, c_ = attention_bwd(dout[:, qs], q[:, qs], k[:, ks], v[:, ks],
                                          out[:, qs], lse[:, :, qs], softmax_scale,
                                          is_causal=(kind == "causal"))
            dq[:, qs] += a
            dk[:, ks] += b_
            dv[:, ks] += c_
    return dq, dk, dv


# ---------------------------------------------------------------------------
# work accounting
# ---------------------------------------------------------------------------

def visible_pairs(lq: int, lk: int, is_causal: bool, window=(-1, -1)) -> int:
    """Number of visible (query, key) pairs of one (batch, head)."""
    left, right = _effective_window(is_causal, window)
    total = 0
    for i in range(lq):
        lo = 0 if left < 0 else max(0, i - left)
        hi = lk - 1 if right < 0 else min(lk - 1, i + right)
        total += max(0, hi - lo + 1)
    return total


def algorithmic_flops(n: int, h: int, lq: int, lk: int, d: int, is_causal: bool,
                      window=(-1, -1)):
    """(fwd, bwd) algorithmic FLOPs: 4*d per visible pair per head for the
    forward (two GEMMs), 2.5x that for the backward. For full and causal
    masks this is 4*n*h*l^2*d (halved for causal, counting l^2/2 pairs)."""
    left, right = _effective_window(is_causal, window)
    if left < 0 and right < 0:
        pairs = lq * lk
    elif is_causal and left < 0:
        pairs = lq * lk / 2.0
    else:
        pairs = visible_pairs(lq, lk, is_causal, window)
    fwd = 4.0 * n * h * d * pairs
    return fwd, 2.5 * fwd


def _selfcheck():  # pragma: no cover - manual sanity entry point
    rng = np.random.default_rng(0)
    q = rng.standard_normal((1, 8, 2, 4))
    k = rng.standard_normal((1, 8, 1, 4))
    v = rng.standard_normal((1, 8, 1, 4))
    o, l = attention_fwd(q, k, v, 1 / math.sqrt(4), True)
    return o, l
