import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


@pytest.fixture(scope="session")
def moelib():
    """The built C-ABI library (built in-tree on first use)."""
    from mixture_experts_layer_tokens_gb300 import build, moe
    build.build()
    return moe.lib()


@pytest.fixture(scope="session")
def cuda_dev(moelib):
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")
