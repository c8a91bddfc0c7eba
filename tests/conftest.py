import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")


@pytest.fixture(scope="session")
def rng():
    import numpy as np
    return np.random.default_rng(1234)


def build_library():
    """Build libcce.so if it is stale (loads build.py by path, see __graft_entry__)."""
    import __graft_entry__
    __graft_entry__._build_module().build()
