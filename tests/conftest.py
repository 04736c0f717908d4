import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: large CPU case")


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def pq():
    """The CUDA library binding; GPU tests fail loudly if it cannot be loaded."""
    if not gpu_available():
        pytest.skip("no CUDA device")
    import gemm_q8_qdot_gb300 as g
    g.load()  # raises if libpq.so is missing
    return g
