"""fp64 CPU oracle: TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library never does.

``sls_oracle`` binds the plain C++ oracle (``sls_oracle.cpp``);
``numpy_oracle`` is a second, independently written numpy oracle that the
tests cross-check against it.
"""
