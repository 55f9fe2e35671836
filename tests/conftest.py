import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def repo_root():
    return ROOT


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Report how many bf16 elements needed the half-ulp rounding allowance
    (results that are bf16 tensors with |ref| >= 4); every other element was
    held to the literal 2e-2."""
    try:
        from helpers import ALLOWANCE_LOG, REPORT_LINES
    except Exception:
        return
    for line in REPORT_LINES:
        terminalreporter.write_line(line)
    if not ALLOWANCE_LOG:
        return
    total = sum(r[1] for r in ALLOWANCE_LOG)
    used = [r for r in ALLOWANCE_LOG if r[2]]
    tr = terminalreporter
    tr.write_line(f"bf16 tolerance: {len(ALLOWANCE_LOG)} comparisons, {total} elements held to 2e-2; "
                  f"{sum(r[2] for r in used)} elements in {len(used)} comparisons needed the half-ulp "
                  f"allowance for bf16 results with |ref| >= 4")
    for name, n, k, mref, merr in used:
        tr.write_line(f"  {name}: {k} of {n} elements, largest |ref| {mref:.3f}, largest err {merr:.3e}")
