import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
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


def pytest_terminal_summary(terminalreporter):
    """Worst and mean |C - C_ref| / bound of every parity comparison made."""
    try:
        from tests._accept import REPORT
    except Exception:  # pragma: no cover
        return
    if not REPORT:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity margins: |C - C_ref| / (4e-3*|C_ref| + 1e-5*T)")
    tr.write_line(f"{'case':44s} {'worst':>8s} {'mean':>9s} {'elements':>10s}")
    for what, (worst, mean, n) in REPORT.items():
        tr.write_line(f"{what[:44]:44s} {worst:8.3f} {mean:9.4f} {n:10d}")
