import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: large CPU work (oracle at full workload size)")


@pytest.fixture(scope="session")
def lib():
    """The C-ABI library, built in-tree when missing (no GPU needed)."""
    from prefill_only_shared_gb300 import build as _build
    _build.ensure_built()
    from prefill_only_shared_gb300 import sp
    return sp


@pytest.fixture(scope="session")
def cuda_dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")
