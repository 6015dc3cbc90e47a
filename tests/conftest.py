import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103) and the built libnvfp4.so")
    config.addinivalue_line("markers", "slow: long CPU test")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def nv():
    """The CUDA binding, built and loaded; skips when no GPU is present."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_weight_only_02_gb300 import binding
    binding.load()
    return binding
