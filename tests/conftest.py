import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running full-size check")


@pytest.fixture(scope="session")
def gpu_lib():
    """The built CUDA library, or a hard failure: GPU tests never fall back."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    from bwd_flashattention_fwd_sm_gb300 import _lib

    return _lib.load()
