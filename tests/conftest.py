import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: CPU test that takes more than a few seconds")


import pytest


@pytest.fixture(scope="session")
def gpu():
    """A CUDA device with the library built; GPU tests fail (not skip) without one."""
    import torch
    from speculative_tree_verify_gb300 import abi, build
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    build.build()
    abi.load()
    return torch.device("cuda")
