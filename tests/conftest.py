import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: large CPU work")


@pytest.fixture(scope="session", autouse=True)
def native_library():
    """Build libtt_denoise.so in-tree if it is missing or older than its sources."""
    from block_wise_diffusion_denoise_b300 import build
    return build.build()
