import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (GB300); runs the CUDA path through the C ABI")
    config.addinivalue_line(
        "markers", "slow: large CPU work (full-size oracle comparisons)")


@pytest.fixture(scope="session")
def libpa():
    """Build (if stale) and load libpa.so; the binding module."""
    from paged_kv_cache_40_gb300 import build as _build
    _build.build()
    import paged_kv_cache_40_gb300 as pa
    pa.lib()
    return pa
