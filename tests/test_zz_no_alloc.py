"""bea_flash_mha_bwd_noalloc: the backward for callers that cannot allocate.

Some callers cannot hand the library a device workspace: a plugin or
foreign-language host that only passes the tensors it owns, or a running
serving loop that must not call cudaMalloc (it can synchronise the device).
This entry point takes its workspace from a fixed array inside the library.
The test calls it through the C ABI twice in a row and compares both results
with the ordinary entry point, within the tolerance the other GPU tests use.
Between the two calls a larger problem runs through the same array, so the
second call starts from stale accumulator rows, D values and log-sum-exps that
differ from its own: every byte it reads must be rewritten by the call itself.
Covered: bf16 at d = 64 and 128, written and accumulated (fp32) gradients, and
the fp32 path.

This file is named so that pytest collects it last; it also passes when run
alone in a fresh process.
"""

import ctypes

import pytest

from helpers import TOL_BF16, TOL_F32

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

OK, WS = 0, -8


def _desc(t):
    from blockwise_exact_attention_gb300 import _lib
    code = _lib.BEA_BF16 if t.dtype == torch.bfloat16 else _lib.BEA_F32
    return _lib.describe(t.data_ptr(), code, t.shape, t.stride())


def _noalloc(lib, tensors, scale, causal, accumulate):
    ds = [_desc(t) for t in tensors]
    stream = torch.cuda.current_stream().cuda_stream
    return lib.bea_flash_mha_bwd_noalloc(*[ctypes.byref(x) for x in ds], scale, int(causal), -1, -1,
                                         int(accumulate), stream)


def _problem(n, l, h, hkv, d, dtype, causal, seed):
    import blockwise_exact_attention_gb300 as bea
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn((n, l, h, d), device="cuda", generator=g).to(dtype)
    k = torch.randn((n, l, hkv, d), device="cuda", generator=g).to(dtype)
    v = torch.randn((n, l, hkv, d), device="cuda", generator=g).to(dtype)
    do = torch.randn((n, l, h, d), device="cuda", generator=g).to(dtype)
    scale = d ** -0.5
    out, lse = bea.flash_mha_fwd(q, k, v, scale, causal)
    return q, k, v, do, out, lse, scale


def _poison(lib):
    """A larger, different problem through the shared array: leaves stale data in the
    accumulator rows, D and log-sum-exp regions the checked call will use."""
    q, k, v, do, out, lse, scale = _problem(1, 1500, 8, 8, 128, torch.bfloat16, False, seed=99)
    grads = [torch.empty(t.shape, dtype=torch.float32, device="cuda") for t in (q, k, v)]
    assert _noalloc(lib, (do, q, k, v, out, lse, *grads), scale, False, False) == OK
    torch.cuda.synchronize()


CASES = [
    # d, accumulate, input dtype
    (128, False, torch.bfloat16),
    (64, False, torch.bfloat16),
    (128, True, torch.bfloat16),
    (64, True, torch.bfloat16),
    (64, False, torch.float32),
]


@pytest.mark.parametrize("d,accumulate,dtype", CASES,
                         ids=[f"d{c[0]}-acc{int(c[1])}-{str(c[2]).split('.')[-1]}" for c in CASES])
def test_noalloc_backward_matches_allocating_backward(d, accumulate, dtype):
    import __graft_entry__ as g
    g.build()
    import blockwise_exact_attention_gb300 as bea
    from blockwise_exact_attention_gb300 import _lib
    lib = _lib.load()

    l = 777 if dtype == torch.bfloat16 else 200
    q, k, v, do, out, lse, scale = _problem(1, l, 4, 2, d, dtype, True, seed=d + 7 * int(accumulate))
    tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_F32
    g0 = [torch.randn(t.shape, device="cuda") for t in (q, k, v)] if accumulate else None
    if accumulate:
        ref = [t.clone() for t in g0]
        bea.flash_mha_bwd(do, q, k, v, out, lse, scale, True, dq=ref[0], dk=ref[1], dv=ref[2], accumulate=True)
    else:
        ref = bea.flash_mha_bwd(do, q, k, v, out, lse, scale, True, grad_dtype=torch.float32)
    torch.cuda.synchronize()

    for call in range(2):
        if call == 1:
            _poison(lib)
        if accumulate:
            dq, dk, dv = (t.clone() for t in g0)
        else:
            dq, dk, dv = (torch.full(t.shape, float("nan"), device="cuda") for t in (q, k, v))
        rc = _noalloc(lib, (do, q, k, v, out, lse, dq, dk, dv), scale, True, accumulate)
        assert rc == OK, lib.bea_status_string(rc)
        torch.cuda.synchronize()
        assert bea.device_status() == 0
        for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            err = float((got - want).abs().max())
            assert err <= tol, f"call {call}: {name} differs by {err}"


def test_noalloc_rejects_problems_larger_than_its_array():
    from blockwise_exact_attention_gb300 import _lib
    lib = _lib.load()
    fake = 0x7F0000000000
    l = 1 << 20
    big = _lib.describe(fake, _lib.BEA_BF16, [1, l, 32, 128], [l * 32 * 128, 32 * 128, 128, 1])
    lse = _lib.describe(fake, _lib.BEA_F32, [1, 32, l], [32 * l, l, 1])
    need = lib.bea_flash_mha_bwd_workspace_size(1, l, 32, 128)
    assert need > 64 * 1024 * 1024
    args = [big] * 5 + [lse] + [big] * 3
    assert lib.bea_flash_mha_bwd_noalloc(*[ctypes.byref(a) for a in args], 0.1, 1, -1, -1, 0, None) == WS
