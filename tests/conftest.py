import os
import sys

import pytest

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if REPO not in sys.path:
    sys.path.insert(0, REPO)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")
    # The C generator and the oracle are plain C and build in a second; build
    # them before any test module imports their ctypes wrappers.
    import __graft_entry__
    from bit_moe_expert_router_gb300 import build as pkg_build
    pkg_build.build_synth()
    __graft_entry__.build_oracle()


@pytest.fixture(scope="session")
def cuda_lib():
    """Path of the built CUDA library (built on demand; nvcc cross-compiles without a GPU)."""
    from bit_moe_expert_router_gb300 import build as pkg_build
    return pkg_build.build_cuda()
