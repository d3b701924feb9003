import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def built_lib():
    """Build libpagedattn.so (nvcc, sm_103a) once per session and load it."""
    import paged_kv_attention_20_gb300 as pka
    pka.build()
    return pka.load()


@pytest.fixture(scope="session")
def cuda_device(built_lib):
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")
