"""Shared helpers of the GPU parity tests (tolerances, uploads, comparisons)."""

from __future__ import annotations

import numpy as np

# Tolerances (stated against the fp64 oracle):
#   bf16 out/dq/dk/dv: max-abs <= 2e-2; an element whose reference is so large
#   that rounding the result itself to bf16 costs more (|ref| >= 4) may add
#   half a bf16 ulp of |ref| — the final cast alone can be that far off.
#   lse: abs <= 1e-3. fp32 path: <= 1e-4 on all outputs. Ring vs single call
#   (both fp32 outputs): <= 1e-3.
TOL_BF16 = 2e-2
TOL_LSE = 1e-3
TOL_F32 = 1e-4
TOL_RING = 1e-3


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.maximum(np.abs(x), 1e-30)
    return 0.5 * np.exp2(np.floor(np.log2(ax)) - 7)


def assert_close_bf16(got: np.ndarray, ref: np.ndarray, name: str, output_is_bf16: bool = True):
    err = np.abs(got.astype(np.float64) - ref)
    bound = TOL_BF16 + (bf16_half_ulp(ref) if output_is_bf16 else 0.0)
    bad = err > bound
    assert not bad.any(), (
        f"{name}: {int(bad.sum())} elements out of tolerance; max err {err.max():.3e} "
        f"at ref {ref.ravel()[np.argmax(err)]:.3e}")
    return float(err.max())


def assert_close(got: np.ndarray, ref: np.ndarray, tol: float, name: str):
    got = got.astype(np.float64)
    both_inf = np.isneginf(got) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):
        err = np.where(both_inf, 0.0, np.abs(got - ref))
    err = np.where(np.isnan(err), np.inf, err)
    assert err.max(initial=0.0) <= tol, f"{name}: max err {err.max():.3e} > {tol:.1e}"
    return float(err.max(initial=0.0))


def to_dev(a: np.ndarray, dtype):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(dtype)


def to_np(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


_INPUT_CACHE: dict = {}


def cached_inputs(name: str) -> dict:
    """make_inputs() of a named workload, generated once per test process."""
    from blockwise_exact_attention_gb300 import workloads
    if name not in _INPUT_CACHE:
        _INPUT_CACHE[name] = workloads.make_inputs(workloads.WORKLOADS[name])
    return _INPUT_CACHE[name]
