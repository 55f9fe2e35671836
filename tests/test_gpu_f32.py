"""The exact fp32 path (SIMT kernels) against the oracle at 1e-4: the tiny
non-causal workload of the measurement plan, plus masks and GQA."""

import numpy as np
import pytest

import oracle
from blockwise_exact_attention_gb300 import workloads

from helpers import TOL_F32, assert_close, to_dev, to_np

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _check(x, scale, causal, window):
    import blockwise_exact_attention_gb300 as bea
    q, k, v, do = (to_dev(x[s], torch.float32) for s in ("q", "k", "v", "dout"))
    out, lse = bea.flash_mha_fwd(q, k, v, scale, causal, window)
    ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], scale, causal, window)
    torch.cuda.synchronize()
    assert_close(to_np(out), ro, TOL_F32, "out")
    assert_close(to_np(lse), rl, TOL_F32, "lse")
    # backward from the oracle's out/lse, rounded to the fp32 that is uploaded
    o_in, l_in = ro.astype(np.float32), rl.astype(np.float32)
    dq, dk, dv = bea.flash_mha_bwd(do, q, k, v, to_dev(o_in, torch.float32), to_dev(l_in, torch.float32), scale,
                                   causal, window)
    torch.cuda.synchronize()
    rdq, rdk, rdv = oracle.attention_bwd(x["dout"], x["q"], x["k"], x["v"], o_in, l_in, scale, causal, window)
    assert_close(to_np(dq), rdq, TOL_F32, "dq")
    assert_close(to_np(dk), rdk, TOL_F32, "dk")
    assert_close(to_np(dv), rdv, TOL_F32, "dv")
    assert bea.device_status() == 0


def test_tiny_fp32_workload():
    w = workloads.WORKLOADS["tiny_fp32"]
    _check(workloads.make_inputs(w), w.softmax_scale, w.is_causal, w.window)


@pytest.mark.parametrize("causal,window", [(True, (-1, -1)), (True, (5, 0)), (False, (7, 3))])
def test_fp32_masks_gqa(causal, window):
    x = workloads.small_case(n=2, l=77, h=4, h_kv=2, d=32, is_causal=causal, window=window, dtype="f32", seed=4)
    _check(x, 0.2, causal, window)


def test_fp32_accumulate():
    import blockwise_exact_attention_gb300 as bea
    x = workloads.small_case(n=1, l=64, h=2, h_kv=1, d=64, dtype="f32", seed=6)
    q, k, v, do = (to_dev(x[s], torch.float32) for s in ("q", "k", "v", "dout"))
    out, lse = bea.flash_mha_fwd(q, k, v, 0.125, True)
    g1 = bea.flash_mha_bwd(do, q, k, v, out, lse, 0.125, True)
    g2 = [t.clone() for t in g1]
    bea.flash_mha_bwd(do, q, k, v, out, lse, 0.125, True, dq=g2[0], dk=g2[1], dv=g2[2], accumulate=True)
    torch.cuda.synchronize()
    for a, b in zip(g1, g2):
        assert torch.allclose(2 * a, b, atol=1e-5)
