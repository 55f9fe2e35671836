"""Parity of ring_merge against the oracle's max/log1p merge (fp64)."""

import numpy as np
import pytest

import oracle
from blockwise_exact_attention_gb300 import workloads

from helpers import assert_close, to_dev, to_np

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _inputs(n, l, h, d, seed, blk_f32):
    rng = np.random.default_rng(seed)
    oa = rng.standard_normal((n, l, h, d)).astype(np.float32)
    ob = rng.standard_normal((n, l, h, d)).astype(np.float32)
    if not blk_f32:
        ob = workloads.round_to_bf16(ob)
    la = (rng.standard_normal((n, h, l)) * 4).astype(np.float32)
    lb = (rng.standard_normal((n, h, l)) * 4).astype(np.float32)
    # dead rows: only a, only b, both
    la[:, :, 0] = -np.inf
    lb[:, :, 1] = -np.inf
    la[:, :, 2] = -np.inf
    lb[:, :, 2] = -np.inf
    oa[:, 0] = 0.0
    ob[:, 1] = 0.0
    return oa, la, ob, lb


@pytest.mark.parametrize("blk_f32", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("final", [False, True])
def test_merge(blk_f32, d, final):
    import blockwise_exact_attention_gb300 as bea
    n, l, h = 2, 333, 3
    oa, la, ob, lb = _inputs(n, l, h, d, 7 + d, blk_f32)
    acc, lacc = to_dev(oa, torch.float32), to_dev(la, torch.float32)
    blk = to_dev(ob, torch.float32 if blk_f32 else torch.bfloat16)
    lblk = to_dev(lb, torch.float32)
    fin = torch.empty((n, l, h, d), dtype=torch.bfloat16, device="cuda") if final else None
    bea.ring_merge(acc, lacc, blk, lblk, out_final=fin)
    torch.cuda.synchronize()
    ro, rl = oracle.merge_max_form(oa, la, ob, lb)
    err = np.abs(to_np(acc) - ro) / (1.0 + np.abs(ro))
    assert err.max() <= 2e-6, err.max()
    assert_close(to_np(lacc), rl, 2e-6 * (1 + np.abs(rl[np.isfinite(rl)]).max()), "lse")
    assert np.all(np.isneginf(to_np(lacc)[:, :, 2]))
    assert np.array_equal(to_np(acc)[:, 2], oa[:, 2].astype(np.float64))  # both dead: untouched
    if final:
        ref_bf = to_np(acc.to(torch.bfloat16))
        assert np.array_equal(to_np(fin), ref_bf)


def test_merge_strided_chunk_views():
    """Merging into a chunk view of a longer sequence touches only that chunk."""
    import blockwise_exact_attention_gb300 as bea
    n, L, h, d, c = 1, 1024, 4, 128, 256
    oa, la, ob, lb = _inputs(n, L, h, d, 3, False)
    acc, lacc = to_dev(oa, torch.float32), to_dev(la, torch.float32)
    blk = to_dev(ob[:, 512:512 + c], torch.bfloat16)
    lblk = to_dev(np.ascontiguousarray(lb[:, :, 512:512 + c]), torch.float32)
    bea.ring_merge(acc.narrow(1, 512, c), lacc.narrow(2, 512, c), blk, lblk)
    torch.cuda.synchronize()
    ro, rl = oracle.merge_max_form(oa[:, 512:512 + c], la[:, :, 512:512 + c], ob[:, 512:512 + c],
                                   lb[:, :, 512:512 + c])
    got = to_np(acc)
    assert np.abs(got[:, 512:512 + c] - ro).max() <= 2e-5
    assert np.array_equal(got[:, :512], oa[:, :512].astype(np.float64))
    assert np.array_equal(got[:, 512 + c:], oa[:, 512 + c:].astype(np.float64))
