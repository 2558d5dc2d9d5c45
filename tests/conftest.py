import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="session", autouse=True)
def tfpa_library():
    """Builds libtfpa.so if it is missing (nvcc cross-compiles without a GPU)."""
    from paged_kv_cache_235_gb300 import binding, build
    if not os.path.exists(binding.LIB_PATH):
        build.build()
    return binding.lib()
