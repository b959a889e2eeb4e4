import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workloads; minutes of oracle time")


@pytest.fixture(scope="session")
def mfsdp():
    """The Python binding of libmfsdp.so, building the library first if needed."""
    from matrix_optimizers_under_gb300 import _build
    _build.ensure_built()
    from matrix_optimizers_under_gb300 import binding
    return binding
