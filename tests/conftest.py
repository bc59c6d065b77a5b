import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def walib():
    """The built C library (nvcc cross-compiles it here and on the GPU host; skipped when up to date)."""
    from chunk_windowed_softmax_gb300 import _build
    _build.build()
    import chunk_windowed_softmax_gb300 as wa
    return wa


@pytest.fixture(scope="session")
def cuda(walib):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return walib
