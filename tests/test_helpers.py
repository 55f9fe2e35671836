"""The parity tolerance itself (CPU): 2e-2 literally below |ref| = 4, the
half-ulp rounding allowance only for bf16 results at |ref| >= 4."""

import numpy as np
import pytest

from helpers import ALLOWANCE_LOG, assert_close_bf16, bf16_half_ulp


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
