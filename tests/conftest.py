import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (runs the sm_103a kernels)")


@pytest.fixture(scope="session")
def gbn():
    """The ctypes binding, building the shared library first if needed."""
    from bwd_bn_pass_gb300 import build, gbnorm
    if not os.path.exists(gbnorm.library_path()):
        build.build_library()
    return gbnorm
