import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


def pytest_sessionstart(session):
    # The CUDA library is built in-tree before any test imports it (nvcc
    # cross-compiles for sm_103a without a GPU); the oracle is built by its
    # own fixture.
    from nvfp4_block_scaled_amax_gb300 import build
    build.build()
