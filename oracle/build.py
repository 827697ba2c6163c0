"""Compile oracle.c into liboracle.so next to it (gcc, OpenMP when present).

Test infrastructure: the oracle is the CPU reference the tests check the
CUDA library against. ``python oracle/build.py`` builds it by hand.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".%d.tmp" % os.getpid()
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        # No OpenMP runtime: the same code, single-threaded.
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
