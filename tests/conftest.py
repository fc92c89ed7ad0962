import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (the sm_103a library on a GB300)")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def zlib():
    """The C library, built in-tree if needed (nvcc cross-compiles without a GPU)."""
    from zero_sharded_mixed_step_gb300 import build
    build.build()
    import zero_sharded_mixed_step_gb300 as zs
    return zs.lib()
