import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def gdn_lib():
    """The CUDA library's Python binding; GPU tests fail loudly if it is missing."""
    if not gpu_available():
        pytest.skip("no CUDA device")
    import hybrid_linear_attention_deltanet_gb300 as gdn
    gdn.load()   # raises if the compiled library is absent
    return gdn
