import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


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
    """How many compared output elements needed more than the 1e-2 figure
    (each within its derived bound, or the test failed) and the largest
    excess."""
    try:
        from tests.helpers import STATS
    except Exception:  # pragma: no cover
        return
    if not STATS["comparisons"]:
        return
    w = STATS["worst"]
    line = (f"parity: {STATS['comparisons']} comparisons, {STATS['elements']} elements, "
            f"{STATS['above_1e2']} above 1e-2")
    if w:
        line += (f"; largest excess {w['excess']:.3g} (error {w['err']:.4g} at exact "
                 f"{w['ref']:.4g}, bound {w['bound']:.4g}) in {w['what']}")
    terminalreporter.write_line(line)
