import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")
    config.addinivalue_line("markers", "slow: large CPU work (full-size sampled parity)")


def pytest_collection_modifyitems(config, items):
    # GPU tests skip cleanly when no device is visible, unless the run asked for them (-m gpu)
    # in which case a missing device is a failure, not a skip.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    markexpr = config.getoption("-m") or ""
    want_gpu = "gpu" in markexpr and "not gpu" not in markexpr
    if has_gpu or want_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
