import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built CUDA library; GPU tests fail loudly if it is missing."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("GPU test collected without a visible CUDA device")
    from exact_attention_forward_attn_gb300 import _lib

    return _lib.load()
