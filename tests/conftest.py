import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running oracle comparisons")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The measured error of every parity check that recorded one, next to
    its gate, so that a shrinking margin shows before a test goes red."""
    try:
        from tests.gpu_util import MARGINS
    except Exception:
        return
    if not MARGINS:
        return
    tr = terminalreporter
    tr.section("parity margins (measured error / gate)")
    worst = sorted(MARGINS, key=lambda m: -m[2] / m[3])
    for test, what, err, gate in worst:
        tr.write_line(f"{err / gate:6.3f}  {err:.3e} / {gate:.1e}  {test} {what}")
