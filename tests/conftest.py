import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: large inputs; minutes of CPU or GPU time")


@pytest.fixture(scope="session")
def golden_dir():
    return GOLDEN


@pytest.fixture(scope="session", autouse=True)
def built_library():
    """Build libpa.so in-tree before the first test when the checkout has none
    (build outputs are not under version control).  The library itself never
    builds on demand: outside the tests a missing build still fails loudly."""
    if not os.path.exists(os.path.join(ROOT, "paged_kv_cache_12_gb300", "libpa.so")):
        from paged_kv_cache_12_gb300 import build

        build.build()
