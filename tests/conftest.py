import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


_REPORT = []  # lines of the run's parity summary


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture
def report(request):
    """Append a line to the run's parity summary, which the terminal report
    prints after the results (also under -q, where captured output of passing
    tests is not shown)."""
    return _REPORT.append


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    if _REPORT:
        terminalreporter.section("parity against the oracle")
        for line in _REPORT:
            terminalreporter.write_line(line)


def pytest_collection_modifyitems(config, items):
    # Without a GPU, gpu-marked tests are skipped rather than failed, so that a
    # bare `pytest` run on a CPU host stays meaningful.
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
