"""fp64 CPU oracle: TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library never does.
"""
from . import sls_oracle  # noqa: F401
