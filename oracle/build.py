"""Compile the C oracle (``kla_oracle.c``) into a shared library.

Test infrastructure only: the library built here is loaded by ``oracle``
(tests, ``__graft_entry__.smoke`` and the bench's CPU-baseline leg), never by
the product path.  Plain ``gcc``; OpenMP when the compiler supports it.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kla_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libkla_oracle.so")


def _compile(openmp: bool) -> subprocess.CompletedProcess:
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-o", LIB, SRC, "-lm"]
    if openmp:
        cmd.insert(1, "-fopenmp")
    return subprocess.run(cmd, capture_output=True, text=True)


def build(force: bool = False) -> str:
    """Build ``libkla_oracle.so`` if missing or older than its source."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    res = _compile(openmp=True)
    if res.returncode != 0:
        res = _compile(openmp=False)
    if res.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + res.stderr)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
