"""Parity of the bf16 tensor-core backward against the fp64 oracle.

The backward's out/lse inputs are the ORACLE's forward results (out rounded
to the uploaded bf16, lse to fp32), never the GPU's, and the oracle backward
consumes exactly those uploaded bits. Small cases span several tiles, a
ragged tail, every mask mode, GQA, both head dims and lq != lk; the full-size
workloads are checked on a subset of heads (all rows of those heads), with the
other heads given inputs whose gradients are exactly zero; the GPU forward is
checked on every row of the same heads against the oracle forward.
"""

import math

import numpy as np
import pytest

import oracle
from blockwise_exact_attention_gb300 import workloads

from helpers import TOL_LSE, assert_close, assert_close_bf16, cached_inputs, to_dev, to_np

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _bwd_inputs(x, scale, causal, window):
    ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], scale, causal, window)
    out_up = workloads.round_to_bf16(ro.astype(np.float32))
    lse_up = rl.astype(np.float32)
    return out_up, lse_up


def run_bwd(x, scale, causal, window, grad_dtype, accumulate=False):
    import blockwise_exact_attention_gb300 as bea
    out_up, lse_up = _bwd_inputs(x, scale, causal, window)
    q, k, v, do = (to_dev(x[s], torch.bfloat16) for s in ("q", "k", "v", "dout"))
    o = to_dev(out_up, torch.bfloat16)
    lse = to_dev(lse_up, torch.float32)
    if accumulate:
        dq0 = torch.randn(q.shape, device="cuda")
        dk0 = torch.randn(k.shape, device="cuda")
        dv0 = torch.randn(v.shape, device="cuda")
        dq, dk, dv = dq0.clone(), dk0.clone(), dv0.clone()
        bea.flash_mha_bwd(do, q, k, v, o, lse, scale, causal, window, dq=dq, dk=dk, dv=dv, accumulate=True)
    else:
        dq, dk, dv = bea.flash_mha_bwd(do, q, k, v, o, lse, scale, causal, window, grad_dtype=grad_dtype)
    torch.cuda.synchronize()
    assert bea.device_status() == 0
    rdq, rdk, rdv = oracle.attention_bwd(x["dout"], x["q"], x["k"], x["v"], out_up, lse_up, scale, causal, window)
    got = [to_np(t) for t in (dq, dk, dv)]
    if accumulate:
        got = [g - to_np(t0) for g, t0 in zip(got, (dq0, dk0, dv0))]
    bf = grad_dtype == torch.bfloat16 and not accumulate
    for name, g, r in zip(("dq", "dk", "dv"), got, (rdq, rdk, rdv)):
        assert_close_bf16(g, r, name, output_is_bf16=bf)


CASES = [
    # n, l, h, hkv, d, causal, window, lk
    (1, 300, 4, 2, 128, True, (-1, -1), None),
    (2, 256, 2, 2, 64, False, (-1, -1), None),
    (1, 517, 3, 1, 128, True, (100, 0), None),
    (1, 384, 2, 2, 128, False, (64, 32), None),
    (1, 200, 2, 1, 64, False, (-1, -1), 333),
    (1, 100, 2, 2, 128, False, (-1, -1), None),
    (1, 640, 8, 2, 64, True, (-1, -1), None),
    (1, 700, 2, 2, 128, True, (0, 0), None),
    (3, 129, 4, 4, 128, True, (-1, -1), None),
    # lq != lk under a mask: the last query aligned with the last key
    (1, 200, 2, 1, 64, True, (-1, -1), 333),
    (1, 300, 2, 2, 128, True, (50, 0), 170),     # the first 130 rows see no key
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:5])) + f"-c{int(c[5])}-w{c[6]}-lk{c[7]}")
def test_bwd_small(case):
    n, l, h, hkv, d, causal, window, lk = case
    x = workloads.small_case(n=n, l=l, h=h, h_kv=hkv, d=d, is_causal=causal, window=window,
                             seed=100 + CASES.index(case), lk=lk)
    run_bwd(x, 1.0 / math.sqrt(d), causal, window, torch.float32)


def test_bwd_bf16_gradients():
    x = workloads.small_case(n=1, l=333, h=4, h_kv=1, d=128, seed=21)
    run_bwd(x, 1.0 / math.sqrt(128), True, (-1, -1), torch.bfloat16)


def test_bwd_bf16_gradients_d64_ragged():
    """bf16 dq/dk/dv at d = 64 with lq = 4k + 3 (the dQ conversion's last group of four rows is partial)."""
    x = workloads.small_case(n=2, l=259, h=4, h_kv=2, d=64, is_causal=False, window=(50, 10), seed=23)
    run_bwd(x, 1.0 / math.sqrt(64), False, (50, 10), torch.bfloat16)


def test_bwd_accumulate():
    x = workloads.small_case(n=1, l=257, h=2, h_kv=2, d=64, seed=22)
    run_bwd(x, 0.125, True, (-1, -1), torch.float32, accumulate=True)


def test_bwd_fp32_out_input():
    """out given in fp32 (the ring accumulator) instead of bf16."""
    import blockwise_exact_attention_gb300 as bea
    x = workloads.small_case(n=1, l=300, h=2, h_kv=1, d=128, seed=23)
    scale = 1.0 / math.sqrt(128)
    ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], scale, True)
    o32, l32 = ro.astype(np.float32), rl.astype(np.float32)
    q, k, v, do = (to_dev(x[s], torch.bfloat16) for s in ("q", "k", "v", "dout"))
    dq, dk, dv = bea.flash_mha_bwd(do, q, k, v, to_dev(o32, torch.float32), to_dev(l32, torch.float32), scale, True,
                                   grad_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = oracle.attention_bwd(x["dout"], x["q"], x["k"], x["v"], o32, l32, scale, True)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert_close_bf16(to_np(g), r, name, output_is_bf16=False)


def test_bwd_is_deterministic():
    import blockwise_exact_attention_gb300 as bea
    x = workloads.small_case(n=1, l=600, h=4, h_kv=2, d=128, seed=24)
    out_up, lse_up = _bwd_inputs(x, 0.09, True, (-1, -1))
    q, k, v, do = (to_dev(x[s], torch.bfloat16) for s in ("q", "k", "v", "dout"))
    o, lse = to_dev(out_up, torch.bfloat16), to_dev(lse_up, torch.float32)
    g1 = bea.flash_mha_bwd(do, q, k, v, o, lse, 0.09, True, grad_dtype=torch.float32)
    g2 = bea.flash_mha_bwd(do, q, k, v, o, lse, 0.09, True, grad_dtype=torch.float32)
    torch.cuda.synchronize()
    # dK/dV are reduced in a fixed order inside one CTA; dQ sums bulk reductions
    # of different CTAs whose order may vary, so it is compared to rounding
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    assert torch.allclose(g1[0], g2[0], atol=1e-5, rtol=0)


# ---- full-size workloads on a subset of heads ---------------------------------------------

FULL = {
    "causal_mha_4k": [5],
    "causal_gqa_8k_rope": [2],     # K/V head 2 -> query heads 8..11
    "swa_32k_d128": [7],
    "full_32k_d64": [3],
    "ring_causal_16k": [9],
}


@pytest.mark.parametrize("name", sorted(FULL))
def test_bwd_full_size_head_subset(name):
    import blockwise_exact_attention_gb300 as bea
    w = workloads.WORKLOADS[name]
    x = cached_inputs(name)
    g = w.h // w.h_kv
    kvs = FULL[name]
    hqs = [kv * g + t for kv in kvs for t in range(g)]
    sub = {"q": x["q"][:, :, hqs], "k": x["k"][:, :, kvs], "v": x["v"][:, :, kvs], "dout": x["dout"][:, :, hqs]}
    ro, rl = oracle.attention_fwd(sub["q"], sub["k"], sub["v"], w.softmax_scale, w.is_causal, w.window)
    out_sub = workloads.round_to_bf16(ro.astype(np.float32))
    lse_sub = rl.astype(np.float32)
    # the other heads: out = 0 and a huge lse make P (and every gradient) exactly 0
    out_full = np.zeros_like(x["q"])
    lse_full = np.full((w.n, w.h, w.l), 1.0e4, dtype=np.float32)
    out_full[:, :, hqs] = out_sub
    lse_full[:, hqs] = lse_sub
    q, k, v, do = (to_dev(x[s], torch.bfloat16) for s in ("q", "k", "v", "dout"))
    hidx = torch.tensor(hqs, device="cuda")
    kidx = torch.tensor(kvs, device="cuda")
    # the GPU forward on every row of these query heads, against the oracle forward just computed
    fo, fl = bea.flash_mha_fwd(q, k, v, w.softmax_scale, w.is_causal, w.window)
    torch.cuda.synchronize()
    assert bea.device_status() == 0
    assert_close_bf16(to_np(fo.index_select(2, hidx)), ro, "fwd out (whole heads)")
    assert_close(to_np(fl.index_select(1, hidx)), rl, TOL_LSE, "fwd lse (whole heads)")
    del fo, fl
    dq, dk, dv = bea.flash_mha_bwd(do, q, k, v, to_dev(out_full, torch.bfloat16), to_dev(lse_full, torch.float32),
                                   w.softmax_scale, w.is_causal, w.window, grad_dtype=torch.float32)
    torch.cuda.synchronize()
    assert bea.device_status() == 0
    rdq, rdk, rdv = oracle.attention_bwd(sub["dout"], sub["q"], sub["k"], sub["v"], out_sub, lse_sub,
                                         w.softmax_scale, w.is_causal, w.window)
    assert_close_bf16(to_np(dq.index_select(2, hidx)), rdq, "dq", output_is_bf16=False)
    assert_close_bf16(to_np(dk.index_select(2, kidx)), rdk, "dk", output_is_bf16=False)
    assert_close_bf16(to_np(dv.index_select(2, kidx)), rdv, "dv", output_is_bf16=False)
    others = [hh for hh in range(w.h) if hh not in hqs]
    if others:
        assert float(dq[:, :, others].abs().max()) == 0.0


# ---- the staged backward (prepare / kv_block / finish) -------------------------------------

def test_staged_bwd_equals_one_call():
    """prepare + kv_block + finish launch the same kernels as flash_mha_bwd."""
    import blockwise_exact_attention_gb300 as bea
    x = workloads.small_case(n=1, l=515, h=4, h_kv=2, d=128, seed=31)
    scale = 1.0 / math.sqrt(128)
    out_up, lse_up = _bwd_inputs(x, scale, True, (-1, -1))
    q, k, v, do = (to_dev(x[s], torch.bfloat16) for s in ("q", "k", "v", "dout"))
    o, lse = to_dev(out_up, torch.bfloat16), to_dev(lse_up, torch.float32)
    ref = bea.flash_mha_bwd(do, q, k, v, o, lse, scale, True, grad_dtype=torch.float32)
    ws = torch.empty(bea.bwd_workspace_bytes(q), dtype=torch.uint8, device="cuda")
    dq, dk, dv = (torch.empty_like(t) for t in ref)
    bea.flash_mha_bwd_prepare(do, o, lse, ws)
    bea.flash_mha_bwd_kv_block(do, q, k, v, dk, dv, scale, True, workspace=ws)
    bea.flash_mha_bwd_finish(dq, scale, workspace=ws)
    torch.cuda.synchronize()
    assert bea.device_status() == 0
    assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
    assert torch.allclose(dq, ref[0], atol=1e-5, rtol=0)


@pytest.mark.parametrize("d", [64, 128])
def test_staged_bwd_accumulates_dq_over_kv_blocks(d):
    """Keys split into two blocks: dQ summed in the workspace over both, dK/dV per block,
    against the oracle backward over all keys."""
    import blockwise_exact_attention_gb300 as bea
    lq, lk = 300, 520
    x = workloads.small_case(n=1, l=lq, h=4, h_kv=2, d=d, seed=32 + d, lk=lk)
    scale = 1.0 / math.sqrt(d)
    out_up, lse_up = _bwd_inputs(x, scale, False, (-1, -1))
    q, k, v, do = (to_dev(x[s], torch.bfloat16) for s in ("q", "k", "v", "dout"))
    o, lse = to_dev(out_up, torch.bfloat16), to_dev(lse_up, torch.float32)
    ws = torch.empty(bea.bwd_workspace_bytes(q), dtype=torch.uint8, device="cuda")
    dq = torch.full(q.shape, 7.0, device="cuda")  # overwritten by finish
    dk = torch.empty(k.shape, device="cuda")
    dv = torch.empty(v.shape, device="cuda")
    cut = 256  # a 16-byte aligned chunk view boundary
    bea.flash_mha_bwd_prepare(do, o, lse, ws)
    for sl in (slice(0, cut), slice(cut, lk)):
        bea.flash_mha_bwd_kv_block(do, q, k[:, sl], v[:, sl], dk[:, sl], dv[:, sl], scale, False, workspace=ws)
    bea.flash_mha_bwd_finish(dq, scale, workspace=ws)
    torch.cuda.synchronize()
    assert bea.device_status() == 0
    rdq, rdk, rdv = oracle.attention_bwd(x["dout"], x["q"], x["k"], x["v"], out_up, lse_up, scale, False)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), (rdq, rdk, rdv)):
        assert_close_bf16(to_np(g), r, name, output_is_bf16=False)


def test_beyond_int32_elements():
    """q, out, dout and dq of 1,052,672 rows x 16 heads x 128 = 2.16e9 elements (past 2^31),
    sliding window (64, 0), GQA 16/2, forward and backward (~27 GB on the device). The last 300
    rows (the largest offsets) and 300 rows at 2^20 against the oracle on a sub-problem that
    holds every key those rows see (key j at query position j - 64): out, lse and dQ of the
    rows, dK/dV of the keys whose every query lies in the sub-problem."""
    import blockwise_exact_attention_gb300 as bea
    L, h, hkv, d, W = 1048576 + 4096, 16, 2, 128, 64
    scale = 1.0 / math.sqrt(d)
    gen = torch.Generator(device="cuda").manual_seed(4242)
    q = torch.randn((1, L, h, d), generator=gen, device="cuda").to(torch.bfloat16)
    k = torch.randn((1, L, hkv, d), generator=gen, device="cuda").to(torch.bfloat16)
    v = torch.randn((1, L, hkv, d), generator=gen, device="cuda").to(torch.bfloat16)
    do = torch.randn((1, L, h, d), generator=gen, device="cuda").to(torch.bfloat16)
    assert q.numel() > 2 ** 31
    out, lse = bea.flash_mha_fwd(q, k, v, scale, True, (W, 0))
    dq, dk, dv = bea.flash_mha_bwd(do, q, k, v, out, lse, scale, True, (W, 0), grad_dtype=torch.float32)
    torch.cuda.synchronize()
    assert bea.device_status() == 0
    assert torch.isfinite(lse).all() and torch.isfinite(out.float()).all()
    for r0 in (L - 300, 1048576 - 150):
        r1, k0 = r0 + 300, r0 - W
        f32 = lambda t: t.float().cpu().numpy()
        qs, ks, vs, dos = f32(q[:, r0:r1]), f32(k[:, k0:r1]), f32(v[:, k0:r1]), f32(do[:, r0:r1])
        ro, rl = oracle.attention_fwd(qs, ks, vs, scale, True, (W, 0), key_offset=-W)
        assert_close_bf16(to_np(out[:, r0:r1]), ro, "out")
        assert_close(to_np(lse[:, :, r0:r1]), rl, TOL_LSE, "lse")
        # the backward from the kernel's own out/lse of these rows
        rdq, rdk, rdv = oracle.attention_bwd(dos, qs, ks, vs, f32(out[:, r0:r1]), f32(lse[:, :, r0:r1]), scale, True,
                                             (W, 0), key_offset=-W)
        assert_close_bf16(to_np(dq[:, r0:r1]), rdq, "dq", output_is_bf16=False)
        # a key is read by the queries up to W after it: complete where those all lie in the rows
        ke = r1 if r1 == L else r1 - W
        assert_close_bf16(to_np(dk[:, r0:ke]), rdk[:, W:W + ke - r0], "dk", output_is_bf16=False)
        assert_close_bf16(to_np(dv[:, r0:ke]), rdv[:, W:W + ke - r0], "dv", output_is_bf16=False)
    del q, k, v, do, out, lse, dq, dk, dv
    torch.cuda.empty_cache()
