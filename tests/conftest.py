import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a B300 GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: large-size case (minutes)")


def pytest_collection_modifyitems(config, items):
    # GPU tests run only when a GPU is present; on a CPU machine they are
    # deselected by -m "not gpu" and skipped otherwise.
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
