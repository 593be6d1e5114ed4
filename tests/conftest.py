import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def cuda_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def gpu():
    """The CUDA library, built in-tree; skips only when there is no GPU at all.

    On a machine with a GPU a missing or broken library is an error, never a
    skip: the GPU tests must run the native code.
    """
    if not cuda_available():
        pytest.skip("no CUDA device")
    import bit_weight_quantized_awq_gb300 as awq
    awq.load_library()
    return awq
