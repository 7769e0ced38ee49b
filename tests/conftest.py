import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    return oracle


def pytest_terminal_summary(terminalreporter):
    """Print the largest error each full-size comparison saw."""
    try:
        import gpu_util
    except ImportError:
        return
    if not gpu_util.ERROR_LOG:
        return
    tr = terminalreporter
    tr.section("max |C_gpu - C_oracle| over every entry")
    for what, n, err, ratio in gpu_util.ERROR_LOG:
        tr.write_line("%-72s %10d entries  max |err| %.3e  max err/allowed %.3f"
                      % (what, n, err, ratio))
