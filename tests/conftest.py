"""Shared pytest set-up: the `gpu` marker and the repository root on sys.path."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (GB300, sm_103a); run with -m gpu")


def have_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


@pytest.fixture(scope="session")
def gpu_lib():
    """The CUDA library's Python binding, built in-tree if needed.  GPU tests
    fail (not skip) when it cannot be loaded: there is no fallback path."""
    if not have_gpu():
        pytest.fail("GPU test selected but torch sees no CUDA device")
    import gated_deltanet_linear_07_gb300 as gdn
    gdn.load()
    return gdn
