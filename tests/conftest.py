import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but torch.cuda.is_available() is False")
    return torch.device("cuda", 0)


@pytest.fixture(scope="session")
def pkv(cuda_device):
    """The CUDA library binding (fails loudly if the extension is not built)."""
    import paged_fp8_kv_03_gb300 as pkv_mod
    pkv_mod.load()
    return pkv_mod
