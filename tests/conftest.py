import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size host checks (seconds to a minute)")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    return oracle.default()


@pytest.fixture(scope="session")
def cuda_dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.fixture(scope="session")
def sc(cuda_dev):
    """The CUDA library binding (built in-tree); fails loudly if it cannot load."""
    import stencil_conv2d_fwd_gb300 as lib
    lib.load()
    return lib
