import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size cases (minutes)")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Prints the error margin of every parity check that ran (value against its bound)."""
    try:
        from gdn_testutil import MARGINS
    except ImportError:
        return
    if not MARGINS:
        return
    tr = terminalreporter
    tr.section("parity margins (error / bound)")
    for test, case, metric, value, bound in MARGINS:
        tr.write_line(f"{test:48s} {case:28s} {metric:44s} {value:.3e} / {bound:.0e}"
                      f"  ({value / bound:5.1%} of bound)")
