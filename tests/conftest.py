import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")
    config.addinivalue_line("markers", "slow: full-size parity case (minutes)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built CUDA library through its Python binding (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected without a CUDA device")
    from qk_norm_rope_gb300 import api
    return api
