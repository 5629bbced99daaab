import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: runs CUDA kernels; needs an sm_103 GPU and the built library")
    config.addinivalue_line("markers", "slow: full-size case (tens of seconds)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, loaded on a GPU.  A GPU test never falls back: a
    missing device or library is an error, not a skip."""
    import torch
    if not torch.cuda.is_available():
        raise RuntimeError("gpu test needs a CUDA device")
    import mlp_gemms_gb300 as mx
    mx.load()
    return mx
