import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA path through the C ABI)")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load_library()


@pytest.fixture(scope="session")
def kvc_library_path():
    """Build libkvc.so if needed (nvcc cross-compiles without a GPU)."""
    from static_kv_cache_gb300 import build
    return build.build()
