import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: CPU test that takes tens of seconds")
    config.addinivalue_line("markers", "full: GPU parity at full workload size (tens of GB, about a minute each)")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle
