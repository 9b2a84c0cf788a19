import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU check")


def pytest_collection_modifyitems(config, items):
    """GPU tests skip without a GPU unless CMD_REQUIRE_GPU=1, which turns the
    skip into a failure (so a machine whose GPU does not come up cannot pass)."""
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu or os.environ.get("CMD_REQUIRE_GPU") == "1":
        return
    skip = pytest.mark.skip(reason="no CUDA GPU visible")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
