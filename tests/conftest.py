import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def golden_path(name: str) -> str:
    return os.path.join(GOLDEN, name)


@pytest.fixture(scope="session")
def kvq():
    """The built package (builds libkvq.so in-tree first if needed)."""
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_fp16_gb300 as pkg
    return pkg


@pytest.fixture(scope="session")
def cuda_dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")
