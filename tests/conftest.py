import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# Lines that parity tests report (rows checked, mismatches, near-tie counts); printed at the end of the run
# even under -q, so that the counts appear in every test log.
PARITY_REPORT = []


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running (large workloads)")


@pytest.fixture
def parity_report():
    return PARITY_REPORT


def pytest_terminal_summary(terminalreporter):
    if PARITY_REPORT:
        terminalreporter.section("parity summary")
        for line in PARITY_REPORT:
            terminalreporter.write_line(line)
