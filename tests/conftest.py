import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload, minutes of oracle time")


@pytest.fixture(scope="session")
def lib():
    """The CUDA library through its Python binding; built on first use."""
    import paged_kv_cache_184_gb300 as pa
    pa.load()
    return pa
