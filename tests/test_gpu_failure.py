"""Failure detection without a GPU fault: a kernel waits on an mbarrier that
nothing arrives on, gives up after its limit, returns normally, and the host
reads BEA_ERR_TIMEOUT from the status word; the context stays usable."""

import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def test_wait_timeout_is_reported_and_context_survives():
    import __graft_entry__ as g
    g.build()
    import blockwise_exact_attention_gb300 as bea
    assert bea.device_status() == 0
    bea.selftest_wait_timeout(20000)          # 20 ms limit
    assert bea.device_status() == -7          # BEA_ERR_TIMEOUT
    assert bea.device_status() == 0           # read clears it
    q = torch.randn((1, 256, 2, 128), device="cuda").to(torch.bfloat16)
    out, lse = bea.flash_mha_fwd(q, q, q, 0.1, True)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all() and bea.device_status() == 0


# Aborts injected into the attention kernels themselves: the first CTA's MMA warp
# behaves as if one of its waits had run out at the given tile. Every other role
# must leave its loop (the named-barrier hand-offs stay matched), the kernel must
# return, the status word must read BEA_ERR_TIMEOUT, and the next clean call must
# give the same result as before.

def _clean_and_aborted(run, tile):
    import blockwise_exact_attention_gb300 as bea
    ref = [t.clone() for t in run()]
    torch.cuda.synchronize()
    assert bea.device_status() == 0
    bea.selftest_inject_abort(tile)
    run()
    torch.cuda.synchronize()
    assert bea.device_status() == -7          # BEA_ERR_TIMEOUT, then cleared
    assert bea.device_status() == 0
    again = run()
    torch.cuda.synchronize()
    assert bea.device_status() == 0
    return ref, again


@pytest.mark.parametrize("tile", [0, 1, 5, 7])
def test_injected_abort_in_forward(tile):
    import __graft_entry__ as g
    g.build()
    import blockwise_exact_attention_gb300 as bea
    gen = torch.Generator().manual_seed(11)
    q, k, v = (torch.randn((1, 1024, 2, 128), generator=gen).to(torch.bfloat16).cuda() for _ in range(3))
    # the first CTA takes the last 256 query rows: key tiles 0..7 under the causal mask
    ref, again = _clean_and_aborted(lambda: bea.flash_mha_fwd(q, k, v, 128 ** -0.5, True), tile)
    for a, b in zip(ref, again):
        assert torch.equal(a, b)


@pytest.mark.parametrize("tile", [0, 1, 9, 15])
def test_injected_abort_in_backward(tile):
    import __graft_entry__ as g
    g.build()
    import blockwise_exact_attention_gb300 as bea
    gen = torch.Generator().manual_seed(12)
    q = torch.randn((1, 1024, 4, 128), generator=gen).to(torch.bfloat16).cuda()
    k, v = (torch.randn((1, 1024, 2, 128), generator=gen).to(torch.bfloat16).cuda() for _ in range(2))
    do = torch.randn((1, 1024, 4, 128), generator=gen).to(torch.bfloat16).cuda()
    out, lse = bea.flash_mha_fwd(q, k, v, 128 ** -0.5, True)
    # the first CTA takes key block 0: 2 query heads x 8 query tiles = 16 iterations
    ref, again = _clean_and_aborted(
        lambda: bea.flash_mha_bwd(do, q, k, v, out, lse, 128 ** -0.5, True, grad_dtype=torch.float32), tile)
    for a, b in zip(ref, again):
        # dq is summed with reductions in any order: equal to rounding
        assert torch.allclose(a, b, rtol=0, atol=1e-5)


@pytest.mark.parametrize("tile", [0, 1, 7])
def test_injected_abort_in_fused_ring_step(tile):
    """The fused ring step: the aborted CTA's producer and V warps stop staging the accumulator
    (their waits on the K/V releases give up with the abort) and its epilogue writes nothing."""
    import __graft_entry__ as g
    g.build()
    import blockwise_exact_attention_gb300 as bea
    gen = torch.Generator().manual_seed(13)
    q, k, v, k2, v2 = (torch.randn((1, 1024, 2, 128), generator=gen).to(torch.bfloat16).cuda() for _ in range(5))
    acc0, lse0 = bea.flash_mha_fwd(q, k2, v2, 128 ** -0.5, True, out_dtype=torch.float32)
    torch.cuda.synchronize()

    def run():
        acc, lse = acc0.clone(), lse0.clone()
        bea.flash_mha_fwd_merge(q, k, v, acc, lse, 128 ** -0.5, True)
        return acc, lse

    ref, again = _clean_and_aborted(run, tile)
    for a, b in zip(ref, again):
        assert torch.equal(a, b)


@pytest.mark.parametrize("tile", [0, 3])
def test_injected_abort_in_ring_call(tile):
    """The library's ring call: the abort lands in its first launch (the step that initialises
    the accumulator); the later steps, chained to it, still run, and the call is repeatable."""
    import __graft_entry__ as g
    g.build()
    import blockwise_exact_attention_gb300 as bea
    gen = torch.Generator().manual_seed(14)
    q, k, v = (torch.randn((1, 2048, 2, 128), generator=gen).to(torch.bfloat16).cuda() for _ in range(3))

    def run():
        acc = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        lse = torch.empty((1, 2, 2048), dtype=torch.float32, device="cuda")
        bea.ring_attention_fwd_steps(q, k, v, acc, lse, 4, 128 ** -0.5, True)
        return acc, lse

    ref, again = _clean_and_aborted(run, tile)
    for a, b in zip(ref, again):
        assert torch.equal(a, b)


@pytest.mark.parametrize("tile", [0, 9])
def test_injected_abort_in_backward_accumulate(tile):
    """The backward adding into fp32 dq/dk/dv: the aborted CTA issues no TMA reduce-adds."""
    import __graft_entry__ as g
    g.build()
    import blockwise_exact_attention_gb300 as bea
    gen = torch.Generator().manual_seed(15)
    q = torch.randn((1, 1024, 4, 128), generator=gen).to(torch.bfloat16).cuda()
    k, v = (torch.randn((1, 1024, 2, 128), generator=gen).to(torch.bfloat16).cuda() for _ in range(2))
    do = torch.randn((1, 1024, 4, 128), generator=gen).to(torch.bfloat16).cuda()
    out, lse = bea.flash_mha_fwd(q, k, v, 128 ** -0.5, True)
    base = [torch.randn(t.shape, generator=gen).cuda() for t in (q, k, v)]

    def run():
        dq, dk, dv = (t.clone() for t in base)
        bea.flash_mha_bwd(do, q, k, v, out, lse, 128 ** -0.5, True, dq=dq, dk=dk, dv=dv, accumulate=True)
        return dq, dk, dv

    ref, again = _clean_and_aborted(run, tile)
    for a, b in zip(ref, again):
        assert torch.allclose(a, b, rtol=0, atol=1e-5)
