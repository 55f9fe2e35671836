"""bea_flash_mha_bwd_noalloc: the backward for callers that cannot allocate.

Some callers cannot hand the library a device workspace: a plugin or
foreign-language host that only passes the tensors it owns, or a running
serving loop that must not call cudaMalloc (it can synchronise the device).
This entry point takes its workspace from a fixed array inside the library.
The test calls it through the C ABI twice in a row (the second call sees the
first call's leftovers in the shared array) and compares both results with
the ordinary entry point, within the tolerance the other GPU tests use.

This file is named so that pytest collects it last; it also passes when run
alone in a fresh process.
"""

import ctypes

import pytest

from helpers import TOL_BF16

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

OK, WS = 0, -8


def _desc(t):
    from blockwise_exact_attention_gb300 import _lib
    code = _lib.BEA_BF16 if t.dtype == torch.bfloat16 else _lib.BEA_F32
    return _lib.describe(t.data_ptr(), code, t.shape, t.stride())


def test_noalloc_backward_matches_allocating_backward():
    import __graft_entry__ as g
    g.build()
    import blockwise_exact_attention_gb300 as bea
    from blockwise_exact_attention_gb300 import _lib
    lib = _lib.load()

    torch.manual_seed(0)
    n, l, h, hkv, d = 1, 777, 4, 2, 128
    scale = d ** -0.5
    q = torch.randn((n, l, h, d), device="cuda").to(torch.bfloat16)
    k = torch.randn((n, l, hkv, d), device="cuda").to(torch.bfloat16)
    v = torch.randn((n, l, hkv, d), device="cuda").to(torch.bfloat16)
    do = torch.randn((n, l, h, d), device="cuda").to(torch.bfloat16)
    out, lse = bea.flash_mha_fwd(q, k, v, scale, True)
    ref = bea.flash_mha_bwd(do, q, k, v, out, lse, scale, True, grad_dtype=torch.float32)
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        dq = torch.full(q.shape, float("nan"), device="cuda")
        dk = torch.full(k.shape, float("nan"), device="cuda")
        dv = torch.full(v.shape, float("nan"), device="cuda")
        ds = [_desc(t) for t in (do, q, k, v, out, lse, dq, dk, dv)]
        rc = lib.bea_flash_mha_bwd_noalloc(*[ctypes.byref(x) for x in ds], scale, 1, -1, -1, 0, stream)
        assert rc == OK, lib.bea_status_string(rc)
        torch.cuda.synchronize()
        assert bea.device_status() == 0
        for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            err = float((got - want).abs().max())
            assert err <= TOL_BF16, f"call {call}: {name} differs by {err}"


def test_noalloc_rejects_problems_larger_than_its_array():
    from blockwise_exact_attention_gb300 import _lib
    lib = _lib.load()
    fake = 0x7F0000000000
    big_q = _lib.describe(fake, _lib.BEA_BF16, [1, 1 << 20, 32, 128], [(1 << 20) * 32 * 128, 32 * 128, 128, 1])
    need = lib.bea_flash_mha_bwd_workspace_size(1, 1 << 20, 32, 128)
    assert need > 64 * 1024 * 1024
    args = [ctypes.byref(big_q)] * 9
    assert lib.bea_flash_mha_bwd_noalloc(*args, 0.1, 1, -1, -1, 0, None) == WS
