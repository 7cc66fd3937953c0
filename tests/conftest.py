import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")


def cuda_ok() -> bool:
    import torch
    return torch.cuda.is_available()


@pytest.fixture(scope="session")
def built():
    """Build libsynth and libmk once per session (no-op when up to date)."""
    import __graft_entry__
    __graft_entry__.build()
    return True
