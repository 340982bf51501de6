import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workloads")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Errors of every GPU-against-oracle comparison, absolute and relative to
    the expected output's RMS (informational; the bounds are absolute)."""
    try:
        from _helpers import REPORT
    except ImportError:
        return
    if not REPORT:
        return
    tr = terminalreporter
    worst = max(REPORT, key=lambda r: r[4])
    tr.write_sep("-", "parity errors (%d comparisons)" % len(REPORT))
    tr.write_line("largest max-abs / RMS: %.3g (%s: max-abs %.3g, RMS %.3g)" % (
        worst[4], worst[0], worst[1], worst[3]))
    tr.write_line("largest mean-abs / RMS: %.3g" % max(r[5] for r in REPORT))
    tr.write_line("largest max-abs: %.3g; largest mean-abs: %.3g" % (
        max(r[1] for r in REPORT), max(r[2] for r in REPORT)))
