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
