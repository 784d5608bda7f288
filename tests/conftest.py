import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (runs through the C-ABI library)")


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.default()


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Parity table of the full-size workloads (requests compared exactly,
    draws near a CDF edge checked by bracket, accept decisions near their
    margin checked for validity only)."""
    try:
        from parity import REPORTS
    except ImportError:
        return
    if not REPORTS:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity against the fp64 oracle (decision margin 1e-5)")
    tr.write_line("%-36s %8s %5s %7s %11s %10s %10s" % (
        "workload", "requests", "bad", "exact", "draw_border", "matching", "borderline"))
    for label, r in REPORTS:
        tr.write_line("%-36s %8d %5d %7d %11d %10d %10d" % (
            label, r["requests"], r["bad"], r["exact"], r["draw_border"],
            r["draw_border_matching"], r["borderline"]))
