"""The parity tolerances themselves (CPU): 2e-2 literally below |ref| = 4, the
half-ulp rounding allowance only for bf16 results at |ref| >= 4, and the
ring-vs-single-call bound against an emulation of the P rounding it covers."""

import numpy as np
import pytest

from helpers import ALLOWANCE_LOG, assert_close_bf16, assert_within, bf16_half_ulp, ring_out_bound


def test_half_ulp_values():
    assert bf16_half_ulp(np.array([1.0]))[0] == 2.0 ** -8
    assert bf16_half_ulp(np.array([4.0]))[0] == 2.0 ** -6
    assert bf16_half_ulp(np.array([-7.9]))[0] == 2.0 ** -6
    assert bf16_half_ulp(np.array([8.0]))[0] == 2.0 ** -5


def test_literal_bound_below_four():
    ref = np.array([3.0, 0.1])
    n0 = len(ALLOWANCE_LOG)
    assert_close_bf16(ref + np.array([0.0199, -0.0199]), ref, "edge")
    with pytest.raises(AssertionError):
        assert_close_bf16(np.array([3.0 + 0.025, 0.1]), ref, "just above")
    del ALLOWANCE_LOG[n0:]


def test_allowance_only_for_bf16_results_at_four_and_above():
    ref = np.array([5.0, 1.0])
    got = np.array([5.0 + 0.03, 1.0])
    n0 = len(ALLOWANCE_LOG)
    assert_close_bf16(got, ref, "bf16 result")           # 0.03 <= 0.02 + 0.0156
    assert ALLOWANCE_LOG[n0][2] == 1                     # counted as needing the allowance
    with pytest.raises(AssertionError):
        assert_close_bf16(got, ref, "fp32 result", output_is_bf16=False)
    with pytest.raises(AssertionError):
        assert_close_bf16(np.array([5.0 + 0.04, 1.0]), ref, "beyond the allowance")
    del ALLOWANCE_LOG[n0:]   # keep this self-test out of the session's allowance report


def test_nan_fails():
    with pytest.raises(AssertionError):
        assert_close_bf16(np.array([np.nan]), np.array([0.0]), "nan")


def _rounded_p_out(s, v, shift):
    """out with P rounded to bf16 under a row maximum raised by `shift` (natural-log units),
    the row sum over the unrounded P: the two ingredients the ring-vs-single bound assumes."""
    from blockwise_exact_attention_gb300.workloads import round_to_bf16
    m = s.max(axis=1, keepdims=True) + shift[:, None]
    p = np.exp(s - m)
    p_hat = round_to_bf16(p.astype(np.float32)).astype(np.float64)
    return (p_hat @ v) / p.sum(axis=1, keepdims=True)


def test_ring_out_bound_covers_p_rounding():
    """Two outputs whose P are rounded to bf16 under different row maxima (as a ring step and
    the single call do) stay within ring_out_bound of each other, and each within half of it
    of the exact output; a bound without the |V| weighting (2^-8 alone) would not hold."""
    rng = np.random.default_rng(5)
    n_rows, n_keys, d = 64, 300, 32
    s = rng.normal(size=(n_rows, n_keys)) * 2.0
    v = np.round(rng.normal(size=(n_keys, d)) * 3.0, 2)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    exact, a_abs = p @ v, p @ np.abs(v)
    bound = ring_out_bound(a_abs)
    o1 = _rounded_p_out(s, v, np.zeros(n_rows))
    o2 = _rounded_p_out(s, v, rng.uniform(0.0, 8.0 * np.log(2.0), size=n_rows))
    assert np.all(np.abs(o1 - exact) <= 0.5 * bound)
    assert np.all(np.abs(o2 - exact) <= 0.5 * bound)
    err, frac = assert_within(o1, o2, bound, "two roundings")
    assert 0.0 < frac <= 1.0
    assert np.abs(o1 - o2).max() > 2.0 ** -8   # a constant bound of 2^-8 would not hold here


def test_assert_within_reports_the_worst_element():
    with pytest.raises(AssertionError, match="1 elements beyond"):
        assert_within(np.array([1.0, 2.0]), np.array([1.0, 2.1]), np.array([0.01, 0.05]), "x")
    with pytest.raises(AssertionError):
        assert_within(np.array([np.nan]), np.array([0.0]), np.array([1.0]), "nan")
