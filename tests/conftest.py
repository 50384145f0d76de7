import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The near-tie counts and test statistics the GPU tests reported
    (parity_util.report), shown even under -q."""
    from parity_util import SUMMARY
    if SUMMARY:
        terminalreporter.section("parity and distribution summary")
        for line in SUMMARY:
            terminalreporter.write_line(line)


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle
