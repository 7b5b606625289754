import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running case")


def pytest_terminal_summary(terminalreporter):
    """Tolerance headroom of every output comparison of the run."""
    try:
        from tests import parity
    except Exception:
        return
    if not parity.REPORT:
        return
    tr = terminalreporter
    tr.section("parity headroom: worst |gpu - oracle| / (atol + rtol |oracle|), 1.0 = tolerance edge")
    for what, ratio, mx, n in parity.REPORT:
        tr.write_line("%-70s %7.4f  max|diff| %.3g  (%d elements)" % (what[:70], ratio, mx, n))
