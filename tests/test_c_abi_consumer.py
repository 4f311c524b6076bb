"""The boundary is a C ABI: a C99 program that includes include/sls.h and
links libsls.so compiles with gcc (-Wall -Werror -pedantic) and gets the
documented status codes from calls that fail validation before any launch.
CPU only."""
import os
import shutil
import subprocess

import pytest

from sparse_long_context_gb300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "sparse_long_context_gb300")


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c99_program_uses_the_abi(lib):
    out_dir = os.path.join(PKG, "_build")     # the package's (git-ignored) build folder
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "abi_consumer")
    cc = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
          os.path.join(ROOT, "tests", "c", "abi_consumer.c"), "-L", PKG, "-lsls", f"-Wl,-rpath,{PKG}",
          "-o", exe]
    r = subprocess.run(cc, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    out = dict(line.split("=", 1) for line in r.stdout.splitlines())
    assert int(out["version"]) == 10000
    assert int(out["select_ws"]) == 2 * 2 * 64 * 4
    assert int(out["null_desc"]) == L.SLS_EINVAL
    assert int(out["null_cache"]) == L.SLS_EINVAL and "k_cache" in out["error"]
    assert int(out["misaligned"]) == L.SLS_EINVAL
    assert int(out["bad_dim"]) == L.SLS_EUNSUPPORTED
    assert int(out["stats_null"]) == L.SLS_EINVAL
