import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads")


@pytest.fixture(scope="session")
def oracle():
    import oracle as _o
    _o._load()
    return _o


@pytest.fixture(scope="session")
def fd():
    """The C-ABI library binding; GPU tests fail loudly if it cannot be loaded."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected without a CUDA device")
    import long_context_decode_split_gb300 as _fd
    _fd.load()
    return _fd
