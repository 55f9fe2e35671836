"""Ring attention replayed as chunk steps on one GPU: forward chunk steps
folded with ring_merge, and chunk-pair backward accumulation, checked against
the single-call kernels (both with fp32 outputs, <= 1e-3) and the oracle."""

import math

import numpy as np
import pytest

import oracle
from blockwise_exact_attention_gb300 import workloads

from helpers import TOL_LSE, TOL_RING, assert_close, assert_close_bf16, cached_inputs, to_dev, to_np

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
    torch.cuda.synchronize()
    assert_close(to_np(ro32), to_np(so32), TOL_RING, "ring vs single out")
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


def test_ring_full_size():
    """[1, 16384, 16, 128] as 8 chunks of 2048: 36 chunk forwards, 28 merges."""
    import blockwise_exact_attention_gb300 as bea
    w = workloads.WORKLOADS["ring_causal_16k"]
    x = cached_inputs("ring_causal_16k")
    q, k, v, do = (to_dev(x[s], torch.bfloat16) for s in ("q", "k", "v", "dout"))
    s = w.softmax_scale
    bea.launches_since_reset(reset=True)
    ro32, rl32 = bea.ring_attention_fwd(q, k, v, w.ring_chunks, s, True, out_dtype=torch.float32,
                                        block_dtype=torch.float32)
    assert bea.launches_since_reset(reset=True) == 36 + 28
    so32, sl32 = bea.flash_mha_fwd(q, k, v, s, True, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert_close(to_np(ro32), to_np(so32), TOL_RING, "ring vs single out (fp32)")
    assert_close(to_np(rl32), to_np(sl32), TOL_RING, "ring vs single lse")
    # the bf16 mode rounds every block to bf16 before the merge (as the pages
    # feed the kernel's q-dtype output into the fp32 accumulator), so its
    # result is held to the bf16 tolerance against the single call
    rob, rlb = bea.ring_attention_fwd(q, k, v, w.ring_chunks, s, True)
    sob, _ = bea.flash_mha_fwd(q, k, v, s, True)
    torch.cuda.synchronize()
    assert float(np.abs(to_np(rob) - to_np(sob)).max()) <= 2e-2
    # sampled rows against the oracle
    rows = np.array([0, 2047, 2048, 4095, 8191, 12000, 16383])
    oo, ol = oracle.attention_fwd(x["q"], x["k"], x["v"], s, True, rows=rows)
    idx = torch.from_numpy(rows).cuda()
    assert_close_bf16(to_np(rob.index_select(1, idx)), oo, "ring out")
    assert_close(to_np(rlb.index_select(2, idx)), ol, TOL_LSE, "ring lse")
    # backward: chunk pairs against one call, from the same (fp32) out/lse
    rg = bea.ring_attention_bwd(do, q, k, v, so32, sl32, w.ring_chunks, s, True)
    sg = bea.flash_mha_bwd(do, q, k, v, so32, sl32, s, True, grad_dtype=torch.float32)
    torch.cuda.synchronize()
    for name, a, b in zip(("dq", "dk", "dv"), rg, sg):
        assert_close(to_np(a), to_np(b), TOL_RING, name + " ring vs single")
    assert bea.device_status() == 0
