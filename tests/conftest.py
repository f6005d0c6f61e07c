import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def repo_root():
    return ROOT


def pytest_terminal_summary(terminalreporter):
    # lines the parity tests report (per-layer errors at full size), printed
    # after the run even in quiet mode
    from tests._util import REPORT
    if REPORT:
        terminalreporter.write_sep("-", "parity report")
        for line in REPORT:
            terminalreporter.write_line(line)
