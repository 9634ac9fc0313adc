import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running case")


GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="session")
def swslib():
    """Builds libsws.so in-tree if it is missing or stale, then loads it."""
    import __graft_entry__
    __graft_entry__.build()
    import sharded_weight_storage_gb300 as S
    return S


def cuda_ok():
    import torch
    return torch.cuda.is_available()
