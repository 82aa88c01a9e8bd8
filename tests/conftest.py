import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def gpu_lib():
    """The CUDA library, loaded through its Python binding; fails loudly if absent."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("gpu test selected but no CUDA device is visible")
    from mxfp4_mixture_experts_top_gb300 import moe
    moe.load()
    return moe
