import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Error margins of the parity tests that recorded them: the bare
    max|dO|/rms(o_ref), the same after each stored value's own rounding
    allowance (the quantity the bound applies to), and the state error."""
    try:
        from kda_testutil import MARGINS
    except ImportError:
        return
    if not MARGINS:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity margins (max|dO|/rms bare, rounding-adjusted; state rel. Frobenius)")
    for label in sorted(MARGINS):
        bare, adj, st = MARGINS[label]
        st_s = "-" if st is None else f"{st:.3e}"
        tr.write_line(f"{label:48s} bare {bare:.4e}  adjusted {adj:.4e}  state {st_s}")
