import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built TreeWY library on a GPU machine (builds it if needed)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gdn_speculative_tree_gb300 import binding
    binding.load()
    return binding


@pytest.fixture(scope="session")
def oracle_pool():
    """The oracle on every host core (worker processes started with spawn,
    which is safe after the GPU has been used)."""
    from oracle.pool import OraclePool
    with OraclePool() as pool:
        yield pool
