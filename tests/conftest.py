import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size parity case (minutes)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """Error of the CUDA outputs against the fully unrounded fp64 oracle
    (information only; the asserted comparison rounds where the layer stores
    bf16)."""
    try:
        from tests._util import EXACT_REPORT
    except Exception:  # pragma: no cover
        return
    if not EXACT_REPORT:
        return
    tr = terminalreporter
    tr.section("error against the unrounded fp64 oracle (information)")
    for name, r, m in EXACT_REPORT:
        tr.write_line(f"{name:60s} rel_l2 {r:.3e}  max_abs {m:.3e}")
