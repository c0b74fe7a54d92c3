import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")
    config.addinivalue_line("markers", "slow: CPU test that takes more than a few seconds")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Prints the parity counts the GPU tests collected (near ties, free-running
    differences with their gaps, worst errors), and writes them as JSON where
    the PARITY_RECORD environment variable names a file."""
    try:
        import parity
    except ImportError:  # pragma: no cover
        return
    if not parity.RECORD:
        return
    import json
    tr = terminalreporter
    tr.section("parity record (CUDA path vs fp64 oracle)")
    for r in parity.RECORD:
        tr.write_line(json.dumps(r, sort_keys=True))
    path = os.environ.get("PARITY_RECORD")
    if path:
        with open(path, "w") as f:
            json.dump(parity.RECORD, f, indent=1, sort_keys=True)
