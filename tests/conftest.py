import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running check (full-size workloads)")


def pytest_collection_modifyitems(config, items):
    # GPU tests fail loudly (not skip) when no GPU is present: the driver selects them with
    # -m gpu only on a GPU machine, and a silent skip there would hide a missing CUDA path.
    pass


def pytest_terminal_summary(terminalreporter):
    from tests import search_report
    for line in search_report.summary_lines():
        terminalreporter.write_line(line)


@pytest.fixture(scope="session")
def oracle():
    from oracle import awq_ref
    return awq_ref
