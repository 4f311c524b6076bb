import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA path)")


@pytest.fixture(scope="session")
def lib():
    """The C-ABI library, built in-tree if missing."""
    from sparse_long_context_gb300 import _lib
    return _lib.load(build_if_missing=True)
