import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built det_gemm library")
    config.addinivalue_line("markers", "slow: large inputs; minutes rather than seconds")


def pytest_collection_modifyitems(config, items):
    # GPU tests without a GPU are skipped here rather than failed, so that
    # `-m "not gpu"` and a bare run both work on a CPU-only machine. With a
    # GPU present they run, and a missing library fails them loudly.
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
