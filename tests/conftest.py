import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the built libdgcanvas")
    config.addinivalue_line("markers", "slow: long CPU-side oracle run")


@pytest.fixture(scope="session")
def lib():
    """The C-ABI library, loaded once per session (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    from canvas_denoising_gb300 import binding
    return binding.load()
