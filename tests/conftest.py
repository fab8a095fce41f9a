import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the library's kernels)")
    config.addinivalue_line("markers", "slow: full-size shapes (minutes)")


@pytest.fixture(scope="session")
def has_gpu():
    import torch
    return torch.cuda.is_available()
