import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def gpu_lib():
    """The C-ABI library on a GPU machine; fails loudly if the build is missing."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("gpu-marked test run without a visible CUDA device")
    from tiled_attention_forward_02_gb300 import attn
    attn.load()  # raises if the shared library was not built
    return attn
