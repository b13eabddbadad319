import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    have_gpu = False
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:
        pass
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """Largest observed error of each compared quantity, relative to its
    stated bar (filled by the parity helpers during the GPU tests)."""
    try:
        import parity
    except Exception:
        return
    if parity.REPORT:
        terminalreporter.write_sep("-", "parity: max observed error / stated bar")
        for k in sorted(parity.REPORT):
            terminalreporter.write_line(f"{k}: {parity.REPORT[k]:.4g}")
