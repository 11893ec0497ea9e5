import os
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 values of a bf16 tensor (any device)."""
    return t.detach().to("cpu").float().double().numpy()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns as uint16."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
