"""Parity of the bf16 tensor-core forward against the fp64 oracle.

Small cases (the oracle finishes in seconds) span several 128-row tiles and a
ragged tail, every mask mode, GQA, both head dims, lq != lk, tiny and empty
sequences, strided inputs and fp32 outputs. The full-size workloads are
checked on sampled query rows, which the oracle computes one by one.
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


def run_case(n, l, h, hkv, d, causal, window, lk=None, seed=0, out_dtype=None):
    import blockwise_exact_attention_gb300 as bea
    x = workloads.small_case(n=n, l=l, h=h, h_kv=hkv, d=d, is_causal=causal, window=window, seed=seed, lk=lk)
    q, k, v = (to_dev(x[s], torch.bfloat16) for s in ("q", "k", "v"))
    scale = 1.0 / math.sqrt(d)
    out, lse = bea.flash_mha_fwd(q, k, v, scale, causal, window, out_dtype=out_dtype)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], scale, causal, window)
    assert_close_bf16(to_np(out), ro, "out", output_is_bf16=out.dtype == torch.bfloat16)
    assert_close(to_np(lse), rl, TOL_LSE, "lse")
    assert bea.device_status() == 0


CASES = [
    # n, l, h, hkv, d, causal, window, lk
    (1, 300, 4, 2, 128, True, (-1, -1), None),
    (2, 256, 2, 2, 64, False, (-1, -1), None),
    (1, 517, 3, 1, 128, True, (100, 0), None),
    (1, 384, 2, 2, 128, False, (64, 32), None),
    (1, 200, 2, 1, 64, False, (-1, -1), 333),
    (1, 100, 2, 2, 128, False, (-1, -1), None),
    (1, 1, 2, 1, 128, True, (-1, -1), None),
    (1, 640, 8, 2, 64, True, (-1, -1), None),
    (1, 700, 2, 2, 128, True, (0, 0), None),
    (1, 260, 2, 2, 64, False, (-1, 3), None),
    (3, 129, 4, 4, 128, True, (-1, -1), None),
    # lq != lk under a mask: the last query aligned with the last key
    (1, 200, 2, 1, 64, True, (-1, -1), 333),
    (1, 300, 2, 2, 128, True, (50, 0), 170),     # the first 130 rows see no key
    (1, 129, 4, 2, 128, False, (16, 8), 300),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:5])) + f"-c{int(c[5])}-w{c[6]}-lk{c[7]}")
def test_fwd_small(case):
    n, l, h, hkv, d, causal, window, lk = case
    run_case(n, l, h, hkv, d, causal, window, lk=lk, seed=CASES.index(case))


def test_fwd_fp32_output():
    run_case(1, 333, 2, 1, 128, True, (-1, -1), out_dtype=torch.float32, seed=5)


def test_fwd_diagonal_window_is_exact():
    import blockwise_exact_attention_gb300 as bea
    x = workloads.small_case(n=1, l=300, h=2, h_kv=2, d=128, seed=9)
    q, k, v = (to_dev(x[s], torch.bfloat16) for s in ("q", "k", "v"))
    out, _ = bea.flash_mha_fwd(q, k, v, 0.1, True, (0, 0))
    torch.cuda.synchronize()
    assert torch.equal(out, v)   # one visible key: P = 1 exactly, out = v bit for bit


def test_fwd_strided_views():
    """q/k/v as head slices of one packed [n, l, h + 2 h_kv, d] buffer."""
    import blockwise_exact_attention_gb300 as bea
    rng = np.random.default_rng(11)
    n, l, h, hkv, d = 1, 290, 4, 2, 128
    packed = workloads.round_to_bf16(rng.standard_normal((n, l, h + 2 * hkv, d), dtype=np.float32))
    P = to_dev(packed, torch.bfloat16)
    q, k, v = P[:, :, :h], P[:, :, h:h + hkv], P[:, :, h + hkv:]
    assert not q.is_contiguous()
    out, lse = bea.flash_mha_fwd(q, k, v, 0.09, True)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_fwd(packed[:, :, :h], packed[:, :, h:h + hkv], packed[:, :, h + hkv:], 0.09, True)
    assert_close_bf16(to_np(out), ro, "out")
    assert_close(to_np(lse), rl, TOL_LSE, "lse")


def test_fwd_empty_keys_and_rows():
    import blockwise_exact_attention_gb300 as bea
    q = torch.zeros((1, 5, 2, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 0, 2, 128), dtype=torch.bfloat16, device="cuda")
    out, lse = bea.flash_mha_fwd(q, k, k, 0.1, False)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))
    q0 = torch.zeros((1, 0, 2, 128), dtype=torch.bfloat16, device="cuda")
    out, lse = bea.flash_mha_fwd(q0, q0, q0, 0.1, True)
    assert out.shape == (1, 0, 2, 128)


def test_fwd_is_deterministic():
    import blockwise_exact_attention_gb300 as bea
    x = workloads.small_case(n=1, l=1000, h=4, h_kv=1, d=128, seed=2)
    q, k, v = (to_dev(x[s], torch.bfloat16) for s in ("q", "k", "v"))
    o1, l1 = bea.flash_mha_fwd(q, k, v, 0.1, True)
    o2, l2 = bea.flash_mha_fwd(q, k, v, 0.1, True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ---- full-size workloads, sampled rows -------------------------------------------------

FULL = ["causal_mha_4k", "causal_gqa_8k_rope", "swa_32k_d128", "full_32k_d64"]


@pytest.mark.parametrize("name", FULL)
def test_fwd_full_size_sampled(name):
    import blockwise_exact_attention_gb300 as bea
    w = workloads.WORKLOADS[name]
    x = cached_inputs(name)
    q, k, v = (to_dev(x[s], torch.bfloat16) for s in ("q", "k", "v"))
    out, lse = bea.flash_mha_fwd(q, k, v, w.softmax_scale, w.is_causal, w.window)
    torch.cuda.synchronize()
    assert bea.device_status() == 0
    rng = np.random.default_rng(123)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, w.l - 1],
                                     rng.choice(w.l, size=24, replace=False)]))
    ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], w.softmax_scale, w.is_causal, w.window, rows=rows)
    idx = torch.from_numpy(rows).cuda()
    assert_close_bf16(to_np(out.index_select(1, idx)), ro, "out")
    assert_close(to_np(lse.index_select(2, idx)), rl, TOL_LSE, "lse")
    # every row has at least its own key, so no output may be non-finite
    assert torch.isfinite(lse).all() and torch.isfinite(out.float()).all()


@pytest.mark.parametrize("d,causal,window,lk", [(128, False, (-1, -1), None), (64, False, (-1, -1), 3700),
                                                (128, True, (300, 0), None), (64, False, (250, 60), None)])
def test_fwd_many_blocks_ragged(d, causal, window, lk):
    """320 CTAs (16 query blocks x 20 query heads over 4 K/V heads), more than two waves, with a
    ragged last query block (4000 rows) and, for d=64, fewer keys than queries. Rows of every
    query block and head against the oracle, and a second call gives the same bits."""
    import blockwise_exact_attention_gb300 as bea
    x = workloads.small_case(n=1, l=4000, h=20, h_kv=4, d=d, is_causal=causal, window=window, seed=140 + d,
                             lk=lk)
    scale = 1.0 / math.sqrt(d)
    q, k, v = (to_dev(x[s], torch.bfloat16) for s in ("q", "k", "v"))
    out, lse = bea.flash_mha_fwd(q, k, v, scale, causal, window)
    torch.cuda.synchronize()
    assert bea.device_status() == 0
    rows = np.unique(np.concatenate([np.arange(0, 4000, 37), np.arange(3840, 4000, 11), [255, 256, 3999]]))
    ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], scale, causal, window, rows=rows)
    idx = torch.from_numpy(rows).cuda()
    assert_close_bf16(to_np(out.index_select(1, idx)), ro, "out")
    assert_close(to_np(lse.index_select(2, idx)), rl, TOL_LSE, "lse")
    # and the same call again
    out2, lse2 = bea.flash_mha_fwd(q, k, v, scale, causal, window)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
