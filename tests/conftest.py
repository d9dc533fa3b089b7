import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _has_gpu():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Report how far GPU outputs strayed past the absolute 1e-2 bar (each
    such element is still within its derived per-element bound, or its test
    failed)."""
    try:
        from tests.gpu_common import STATS
    except Exception:
        return
    if not STATS["elements"]:
        return
    line = (f"parity: {STATS['elements']} output elements compared with the oracle; "
            f"{STATS['above_abs']} above the absolute 1e-2")
    if STATS["worst"] is not None:
        ratio, err, ref, bound, what = STATS["worst"]
        line += f"; worst {err:.3e} ({ratio:.2f} x 1e-2) at ref {ref:.4f}, bound {bound:.3e} [{what}]"
    terminalreporter.write_line(line)
