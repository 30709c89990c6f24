import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: large-configuration parity case")


@pytest.fixture(scope="session")
def loong_lib():
    """The built C-ABI library (built in-tree on first use)."""
    from head_context_attention_gb300 import build, ops
    build.build()
    return ops.lib()


@pytest.fixture(scope="session")
def cuda_device(loong_lib):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")
