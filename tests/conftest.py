import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running (full-size model)")


@pytest.fixture(scope="session")
def tiny_bits():
    from dualar_inputs import TINY, generators
    return generators.make_weights(TINY, seed=0)


@pytest.fixture(scope="session")
def tiny_oracle(tiny_bits):
    from dualar_inputs import TINY
    from oracle import DualAROracle
    return DualAROracle(TINY, tiny_bits, max_pos=4096)
