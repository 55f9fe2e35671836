"""Ring attention replayed as chunk steps on one GPU: forward chunk steps
folded with ring_merge or with the fused ring step (flash_mha_fwd_merge), and
chunk-pair backward accumulation, checked against the single-call kernels
(both with fp32 outputs, <= 1e-3) and the oracle."""

import math

import numpy as np
import pytest

import oracle
from blockwise_exact_attention_gb300 import workloads

from helpers import (TOL_LSE, TOL_RING, assert_close, assert_close_bf16, assert_within, cached_inputs, report,
                     ring_out_bound, to_dev, to_np)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def test_schedule_matches_oracle():
    from blockwise_exact_attention_gb300 import chunk_schedule
    for n in (1, 3, 8):
        for c in (True, False):
            assert chunk_schedule(n, c) == oracle.ring_chunk_schedule(n, c)


@pytest.mark.parametrize("causal", [True, False])
def test_ring_small(causal):
    import blockwise_exact_attention_gb300 as bea
    x = workloads.small_case(n=1, l=1024, h=4, h_kv=2, d=128, is_causal=causal, seed=31)
    scale = 1.0 / math.sqrt(128)
    q, k, v, do = (to_dev(x[s], torch.bfloat16) for s in ("q", "k", "v", "dout"))
    ro32, rl32 = bea.ring_attention_fwd(q, k, v, 4, scale, causal, out_dtype=torch.float32,
                                        block_dtype=torch.float32)
    so32, sl32 = bea.flash_mha_fwd(q, k, v, scale, causal, out_dtype=torch.float32)
    rob, rlb = bea.ring_attention_fwd(q, k, v, 4, scale, causal)
    # the library's ring call: the bf16 result is exactly the cast of its fp32 accumulator
    acc = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    lacc = torch.empty((1, 4, 1024), dtype=torch.float32, device="cuda")
    fin = torch.empty_like(q)
    bea.ring_attention_fwd_steps(q, k, v, acc, lacc, 4, scale, causal, out_final=fin)
    torch.cuda.synchronize()
    assert torch.equal(fin, acc.to(torch.bfloat16)) and torch.equal(fin, rob) and torch.equal(lacc, rlb)
    a_abs, _ = oracle.attention_fwd(x["q"], x["k"], np.abs(x["v"]), scale, causal)
    assert_within(to_np(ro32), to_np(so32), ring_out_bound(a_abs), "ring vs single out")
    assert_close(to_np(rl32), to_np(sl32), TOL_RING, "ring vs single lse")
    oo, ol = oracle.ring_fwd_replay(x["q"], x["k"], x["v"], scale, 4, causal)
    assert_close_bf16(to_np(rob), oo, "ring out (bf16)")
    assert_close(to_np(rlb), ol, TOL_LSE, "ring lse")
    # backward over chunk pairs, from the oracle's out/lse
    o_up = workloads.round_to_bf16(oo.astype(np.float32))
    l_up = ol.astype(np.float32)
    o, lse = to_dev(o_up, torch.bfloat16), to_dev(l_up, torch.float32)
    rg = bea.ring_attention_bwd(do, q, k, v, o, lse, 4, scale, causal)
    sg = bea.flash_mha_bwd(do, q, k, v, o, lse, scale, causal, grad_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = oracle.ring_bwd_replay(x["dout"], x["q"], x["k"], x["v"], o_up, l_up, scale, 4, causal)
    for name, a, b, r in zip(("dq", "dk", "dv"), rg, sg, ref):
        assert_close(to_np(a), to_np(b), TOL_RING, name + " ring vs single")
        assert_close_bf16(to_np(a), r, name, output_is_bf16=False)
    assert bea.device_status() == 0


def _abs_attention(q, k, v, scale, row_block=4096):
    """A = sum_j p_j |v_j| for causal attention (the attention output of |V|), by plain torch
    fp32 ops one head and row block at a time; it scales the ring-vs-single bound only."""
    n, l, h, d = q.shape
    g = h // k.shape[2]
    out = np.empty((n, l, h, d), dtype=np.float64)
    keys = torch.arange(l, device=q.device)
    for b in range(n):
        for hq in range(h):
            kh, vh = k[b, :, hq // g].float(), v[b, :, hq // g].float().abs()
            for r0 in range(0, l, row_block):
                r1 = min(l, r0 + row_block)
                s_ = (q[b, r0:r1, hq].float() @ kh[:r1].T) * scale
                rows = torch.arange(r0, r1, device=q.device)[:, None]
                s_ = s_.masked_fill(keys[None, :r1] > rows, float("-inf"))
                out[b, r0:r1, hq] = (torch.softmax(s_, dim=1) @ vh[:r1]).double().cpu().numpy()
    return out


def test_ring_full_size():
    """[1, 16384, 16, 128] as 8 chunks of 2048: the 36 chunk-pair forwards and 28 merges run as one
    batched call per ring step (8 forwards + 7 merges)."""
    import blockwise_exact_attention_gb300 as bea
    w = workloads.WORKLOADS["ring_causal_16k"]
    x = cached_inputs("ring_causal_16k")
    q, k, v, do = (to_dev(x[s], torch.bfloat16) for s in ("q", "k", "v", "dout"))
    s = w.softmax_scale
    bea.launches_since_reset(reset=True)
    ro32, rl32 = bea.ring_attention_fwd(q, k, v, w.ring_chunks, s, True, out_dtype=torch.float32,
                                        block_dtype=torch.float32)
    assert bea.launches_since_reset(reset=True) == 8 + 7
    so32, sl32 = bea.flash_mha_fwd(q, k, v, s, True, out_dtype=torch.float32)
    torch.cuda.synchronize()
    # both sides against the oracle on sampled rows, reported next to their difference: the two
    # round P to bf16 under different running maxima, so each carries its own rounding error
    rows = np.array([0, 1, 2047, 2048, 2049, 4095, 6000, 8191, 8192, 12000, 14336, 16383])
    oo, ol = oracle.attention_fwd(x["q"], x["k"], x["v"], s, True, rows=rows)
    idx = torch.from_numpy(rows).cuda()
    e_ring = assert_close_bf16(to_np(ro32.index_select(1, idx)), oo, "ring out (fp32) vs oracle", output_is_bf16=False)
    e_single = assert_close_bf16(to_np(so32.index_select(1, idx)), oo, "single out (fp32) vs oracle",
                                 output_is_bf16=False)
    diff_rows = float((ro32.index_select(1, idx) - so32.index_select(1, idx)).abs().max())
    bound = ring_out_bound(_abs_attention(q, k, v, s))
    diff, frac = assert_within(to_np(ro32), to_np(so32), bound, "ring vs single out (fp32)")
    report(f"[ring 16k] max |ring - single| {diff:.3e} over all rows, at most {frac:.2f} of its P-rounding "
          f"bound ({diff_rows:.3e} on the sampled rows); on the sampled rows ring vs oracle {e_ring:.3e}, "
          f"single vs oracle {e_single:.3e}")
    assert_close(to_np(rl32), to_np(sl32), TOL_RING, "ring vs single lse")
    fo32, fl32 = bea.ring_attention_fwd(q, k, v, w.ring_chunks, s, True, out_dtype=torch.float32, fused=True)
    torch.cuda.synchronize()
    assert_within(to_np(fo32), to_np(so32), bound, "fused ring vs single out (fp32)")
    assert_close(to_np(fl32), to_np(sl32), TOL_RING, "fused ring vs single lse")
    del fo32, fl32
    # the bf16 result (fused ring steps, cast at the last step) is held to the
    # bf16 tolerance against the single call
    bea.launches_since_reset(reset=True)
    rob, rlb = bea.ring_attention_fwd(q, k, v, w.ring_chunks, s, True)
    # fused, one library call: one launch per causal ring step, the bf16 cast of the chunk that
    # ends at a step written by that step's launch (no merge launches)
    assert bea.launches_since_reset(reset=True) == 8
    del bound
    sob, _ = bea.flash_mha_fwd(q, k, v, s, True)
    torch.cuda.synchronize()
    assert float(np.abs(to_np(rob) - to_np(sob)).max()) <= 2e-2
    # sampled rows against the oracle
    assert_close_bf16(to_np(rob.index_select(1, idx)), oo, "ring out")
    assert_close(to_np(rlb.index_select(2, idx)), ol, TOL_LSE, "ring lse")
    # backward: chunk pairs against one call, from the same (fp32) out/lse
    rg = bea.ring_attention_bwd(do, q, k, v, so32, sl32, w.ring_chunks, s, True)
    sg = bea.flash_mha_bwd(do, q, k, v, so32, sl32, s, True, grad_dtype=torch.float32)
    torch.cuda.synchronize()
    for name, a, b in zip(("dq", "dk", "dv"), rg, sg):
        assert_close(to_np(a), to_np(b), TOL_RING, name + " ring vs single")
    assert bea.device_status() == 0


# ---- the fused ring step --------------------------------------------------------------------

@pytest.mark.parametrize("d", [64, 128])
def test_fwd_merge_two_key_blocks(d):
    """Forward of keys [0, 256) into an fp32 accumulator, then the fused step with keys
    [256, 520): equals attention over all keys (oracle), and out_final is its bf16 cast."""
    import blockwise_exact_attention_gb300 as bea
    lq, lk, cut = 300, 520, 256
    x = workloads.small_case(n=1, l=lq, h=4, h_kv=2, d=d, is_causal=False, seed=40 + d, lk=lk)
    scale = 1.0 / math.sqrt(d)
    q, k, v = (to_dev(x[s_], torch.bfloat16) for s_ in ("q", "k", "v"))
    acc, lse = bea.flash_mha_fwd(q, k[:, :cut], v[:, :cut], scale, False, out_dtype=torch.float32)
    fin = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    bea.flash_mha_fwd_merge(q, k[:, cut:], v[:, cut:], acc, lse, scale, False, out_final=fin)
    torch.cuda.synchronize()
    assert bea.device_status() == 0
    ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], scale, False)
    assert_close_bf16(to_np(acc), ro, "merged out", output_is_bf16=False)
    assert_close(to_np(lse), rl, TOL_LSE, "merged lse")
    assert torch.equal(fin, acc.to(torch.bfloat16))
    # the same fold through the oracle's merge of the two blocks
    oa, la = oracle.attention_fwd(x["q"], x["k"][:, :cut], x["v"][:, :cut], scale, False)
    ob, lb = oracle.attention_fwd(x["q"], x["k"][:, cut:], x["v"][:, cut:], scale, False)
    om, lm = oracle.merge_max_form(oa, la, ob, lb)
    assert_close_bf16(to_np(acc), om, "merged out vs oracle merge", output_is_bf16=False)


def test_fwd_merge_minus_inf_rows():
    """Accumulator rows at lse = -inf take the block exactly; an empty block leaves the
    accumulator unchanged (both -inf: unchanged, lse stays -inf)."""
    import blockwise_exact_attention_gb300 as bea
    x = workloads.small_case(n=1, l=200, h=2, h_kv=1, d=128, is_causal=False, seed=45)
    scale = 1.0 / math.sqrt(128)
    q, k, v = (to_dev(x[s_], torch.bfloat16) for s_ in ("q", "k", "v"))
    ref, ref_l = bea.flash_mha_fwd(q, k, v, scale, False, out_dtype=torch.float32)
    acc = torch.randn(q.shape, device="cuda")
    lse = torch.full((1, 2, 200), float("-inf"), device="cuda")
    bea.flash_mha_fwd_merge(q, k, v, acc, lse, scale, False)
    torch.cuda.synchronize()
    assert torch.equal(acc, ref) and torch.equal(lse, ref_l)
    acc2 = torch.randn(q.shape, device="cuda")
    keep = acc2.clone()
    lse2 = torch.full((1, 2, 200), float("-inf"), device="cuda")
    empty = torch.zeros((1, 0, 1, 128), dtype=torch.bfloat16, device="cuda")
    bea.flash_mha_fwd_merge(q, empty, empty, acc2, lse2, scale, False)
    torch.cuda.synchronize()
    assert torch.equal(acc2, keep) and bool(torch.isneginf(lse2).all())
    assert bea.device_status() == 0


@pytest.mark.parametrize("causal", [True, False])
def test_ring_fused_equals_unfused(causal):
    """The fused ring step computes exactly the forward + ring_merge of fp32 blocks (to fp32
    rounding), with one batched launch per ring step; against the oracle it holds the bf16-path
    tolerance. (Ring and single call round P to bf16 under different row maxima; their
    difference is held to the bound that rounding allows in the other ring tests.)"""
    import blockwise_exact_attention_gb300 as bea
    x = workloads.small_case(n=1, l=1536, h=4, h_kv=1, d=128, is_causal=causal, seed=46)
    scale = 1.0 / math.sqrt(128)
    q, k, v = (to_dev(x[s_], torch.bfloat16) for s_ in ("q", "k", "v"))
    bea.launches_since_reset(reset=True)
    fo, fl = bea.ring_attention_fwd(q, k, v, 6, scale, causal, out_dtype=torch.float32, fused=True)
    # one batched call per ring step (non-causal: the wrapped pairs of a step are a second call)
    assert bea.launches_since_reset(reset=True) == (6 if causal else 11)
    uo, ul = bea.ring_attention_fwd(q, k, v, 6, scale, causal, out_dtype=torch.float32, block_dtype=torch.float32)
    torch.cuda.synchronize()
    assert_close(to_np(fo), to_np(uo), 1e-5, "fused vs unfused out")
    assert_close(to_np(fl), to_np(ul), 1e-5, "fused vs unfused lse")
    oo, ol = oracle.ring_fwd_replay(x["q"], x["k"], x["v"], scale, 6, causal)
    assert_close_bf16(to_np(fo), oo, "fused ring out", output_is_bf16=False)
    assert_close(to_np(fl), ol, TOL_LSE, "fused ring lse")
    assert bea.device_status() == 0


# ---- the window-aware ring ------------------------------------------------------------------

@pytest.mark.parametrize("causal,window", [(True, (700, 0)), (False, (300, 200)), (True, (0, 0))])
def test_ring_windowed(causal, window):
    """Ring steps masked by sequence position: every live chunk pair gets its key offset,
    pairs outside the window are skipped; forward and backward against the oracle's windowed
    ring replay and against the single call."""
    import blockwise_exact_attention_gb300 as bea
    x = workloads.small_case(n=1, l=2048, h=4, h_kv=2, d=128, is_causal=causal, window=window, seed=60)
    scale = 1.0 / math.sqrt(128)
    q, k, v, do = (to_dev(x[s_], torch.bfloat16) for s_ in ("q", "k", "v", "dout"))
    ro, rl = bea.ring_attention_fwd(q, k, v, 8, scale, causal, out_dtype=torch.float32, window_size=window)
    so, sl = bea.flash_mha_fwd(q, k, v, scale, causal, window, out_dtype=torch.float32)
    torch.cuda.synchronize()
    oo, ol = oracle.ring_fwd_replay(x["q"], x["k"], x["v"], scale, 8, causal, window)
    assert_close_bf16(to_np(ro), oo, "windowed ring out", output_is_bf16=False)
    assert_close(to_np(rl), ol, TOL_LSE, "windowed ring lse")
    assert_close_bf16(to_np(ro), to_np(so).astype(np.float64), "windowed ring vs single", output_is_bf16=False)
    # backward from the oracle's out/lse, against the oracle's windowed ring backward
    o_up = workloads.round_to_bf16(oo.astype(np.float32))
    l_up = ol.astype(np.float32)
    o, lse = to_dev(o_up, torch.bfloat16), to_dev(l_up, torch.float32)
    rg = bea.ring_attention_bwd(do, q, k, v, o, lse, 8, scale, causal, window)
    torch.cuda.synchronize()
    ref = oracle.ring_bwd_replay(x["dout"], x["q"], x["k"], x["v"], o_up, l_up, scale, 8, causal, window)
    for name, a, r in zip(("dq", "dk", "dv"), rg, ref):
        assert_close_bf16(to_np(a), r, name, output_is_bf16=False)
    assert bea.device_status() == 0


# ---- the library's ring call: batches, and the bf16 cast at each chunk's last live step ----

@pytest.mark.parametrize("causal,window", [(True, (-1, -1)), (False, (300, 200)), (False, (-1, 100))])
def test_ring_call_batches_and_final_cast(causal, window):
    """Two batch rows (run one after another), 8 chunks of 128: the fp32 result against the
    single call (within the P-rounding bound) and the oracle's windowed ring replay; the bf16 result is exactly the
    cast of the fp32 accumulator even where the chunks' last live steps differ within a step."""
    import blockwise_exact_attention_gb300 as bea
    n, l, h, hkv, d, C = 2, 1024, 4, 2, 128, 8
    x = workloads.small_case(n=n, l=l, h=h, h_kv=hkv, d=d, is_causal=causal, window=window, seed=77)
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (to_dev(x[s_], torch.bfloat16) for s_ in ("q", "k", "v", "dout"))
    acc = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty((n, h, l), dtype=torch.float32, device="cuda")
    fin = torch.empty_like(q)
    bea.ring_attention_fwd_steps(q, k, v, acc, lse, C, scale, causal, window, out_final=fin)
    so, sl = bea.flash_mha_fwd(q, k, v, scale, causal, window, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert bea.device_status() == 0
    assert torch.equal(fin, acc.to(torch.bfloat16))
    a_abs, _ = oracle.attention_fwd(x["q"], x["k"], np.abs(x["v"]), scale, causal, window)
    assert_within(to_np(acc), to_np(so), ring_out_bound(a_abs), "ring call vs single out")
    assert_close(to_np(lse), to_np(sl), TOL_RING, "ring call vs single lse")
    oo, ol = oracle.ring_fwd_replay(x["q"], x["k"], x["v"], scale, C, causal, window)
    assert_close_bf16(to_np(acc), oo, "ring call out vs oracle", output_is_bf16=False)
    assert_close(to_np(lse), ol, TOL_LSE, "ring call lse vs oracle")
    # backward, from the oracle's out/lse, against the oracle's ring backward and the single call
    o_up = workloads.round_to_bf16(oo.astype(np.float32))
    l_up = ol.astype(np.float32)
    o, lt = to_dev(o_up, torch.bfloat16), to_dev(l_up, torch.float32)
    rg = bea.ring_attention_bwd(do, q, k, v, o, lt, C, scale, causal, window)
    sg = bea.flash_mha_bwd(do, q, k, v, o, lt, scale, causal, window, grad_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = oracle.ring_bwd_replay(x["dout"], x["q"], x["k"], x["v"], o_up, l_up, scale, C, causal, window)
    for name, a, b_, r in zip(("dq", "dk", "dv"), rg, sg, ref):
        assert_close(to_np(a), to_np(b_), TOL_RING, name + " ring call vs single")
        assert_close_bf16(to_np(a), r, name + " ring call", output_is_bf16=False)
    assert bea.device_status() == 0


# ---- chunks that are not a multiple of the 128-row tiles ------------------------------------

@pytest.mark.parametrize("d,causal,window", [(128, True, (-1, -1)), (64, False, (200, 100)), (128, True, (300, 0))])
def test_ring_ragged_chunks(d, causal, window):
    """Chunks of 120 rows: each chunk's last 128-row tile runs past its end into the next chunk,
    so the fused forward's accumulator stores and the ring backward's dK/dV additions must stop
    at the chunk's end (neighbouring chunks keep their own rows). Forward and backward against the
    oracle's ring replay and the single call."""
    import blockwise_exact_attention_gb300 as bea
    n, C, c, h, hkv = 1, 8, 120, 4, 2
    l = C * c
    x = workloads.small_case(n=n, l=l, h=h, h_kv=hkv, d=d, is_causal=causal, window=window, seed=90 + d)
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (to_dev(x[s_], torch.bfloat16) for s_ in ("q", "k", "v", "dout"))
    acc = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty((n, h, l), dtype=torch.float32, device="cuda")
    fin = torch.empty_like(q)
    bea.ring_attention_fwd_steps(q, k, v, acc, lse, C, scale, causal, window, out_final=fin)
    so, sl = bea.flash_mha_fwd(q, k, v, scale, causal, window, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert bea.device_status() == 0
    assert torch.equal(fin, acc.to(torch.bfloat16))
    a_abs, _ = oracle.attention_fwd(x["q"], x["k"], np.abs(x["v"]), scale, causal, window)
    assert_within(to_np(acc), to_np(so), ring_out_bound(a_abs), "ragged ring vs single out")
    assert_close(to_np(lse), to_np(sl), TOL_RING, "ragged ring vs single lse")
    oo, ol = oracle.ring_fwd_replay(x["q"], x["k"], x["v"], scale, C, causal, window)
    assert_close_bf16(to_np(acc), oo, "ragged ring out vs oracle", output_is_bf16=False)
    assert_close(to_np(lse), ol, TOL_LSE, "ragged ring lse vs oracle")
    o_up = workloads.round_to_bf16(oo.astype(np.float32))
    l_up = ol.astype(np.float32)
    o, lt = to_dev(o_up, torch.bfloat16), to_dev(l_up, torch.float32)
    rg = bea.ring_attention_bwd(do, q, k, v, o, lt, C, scale, causal, window)
    sg = bea.flash_mha_bwd(do, q, k, v, o, lt, scale, causal, window, grad_dtype=torch.float32)
    torch.cuda.synchronize()
    assert bea.device_status() == 0
    ref = oracle.ring_bwd_replay(x["dout"], x["q"], x["k"], x["v"], o_up, l_up, scale, C, causal, window)
    for name, a, b_, r in zip(("dq", "dk", "dv"), rg, sg, ref):
        assert_close(to_np(a), to_np(b_), TOL_RING, name + " ragged ring vs single")
        assert_close_bf16(to_np(a), r, name + " ragged ring", output_is_bf16=False)
