"""Builds the C++ oracle (sls_oracle.cpp) into oracle/libslsoracle.so.

TEST INFRASTRUCTURE ONLY.  Plain g++ (C++17, -O2, no target-specific
flags, so that it builds the same on x86-64 and Arm hosts).  build() is also
used by the mutation check to compile planted-mistake variants of the source
into a temporary directory.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "sls_oracle.cpp")
LIB = os.path.join(HERE, "libslsoracle.so")
FLAGS = ["-std=c++17", "-O2", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-Wall", "-Wextra"]


def cxx() -> str:
    for cand in (os.environ.get("CXX"), shutil.which("g++"), shutil.which("c++")):
        if cand:
            return cand
    raise RuntimeError("no C++ compiler found: g++ is needed to build the oracle")


def build(src: str = SOURCE, out: str = LIB, force: bool = False, text: str | None = None,
          opt: str = "-O2") -> str:
    """Compile `src` (or the given source `text`) into the shared library
    `out`; skipped while `out` is newer than `src`.  Returns `out`."""
    if text is None and not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".{os.getpid()}.tmp"
    flags = [f if f != "-O2" else opt for f in FLAGS]
    if text is None:
        cmd = [cxx(), *flags, src, "-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
    else:
        cmd = [cxx(), *flags, "-x", "c++", "-", "-o", tmp]
        r = subprocess.run(cmd, input=text, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"oracle build failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
