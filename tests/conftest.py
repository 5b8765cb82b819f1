import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")


def cuda_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def gda():
    """The CUDA library's Python binding; GPU tests fail loudly if it is missing."""
    if not cuda_available():
        pytest.skip("no CUDA device")
    import gated_gqa_attention_gb300 as g
    g.load()  # raises if the shared library is absent
    return g
