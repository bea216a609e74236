"""Compile the plain-C oracle into a shared library with gcc.

Test infrastructure: the library built here is loaded only by the
test-suite, the package smoke check and the benchmark's CPU baseline.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "pkv_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIBRARY = os.path.join(BUILD_DIR, "liboracle.so")


def build(force: bool = False) -> str:
    """Build ``oracle/_build/liboracle.so`` (OpenMP, -O2, no fast-math)."""
    if (not force and os.path.exists(LIBRARY)
            and os.path.getmtime(LIBRARY) >= os.path.getmtime(SOURCE)):
        return LIBRARY
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = LIBRARY + f".tmp{os.getpid()}"
    # -ffp-contract=off keeps every product and sum a separately rounded
    # binary64 operation, exactly as written in the source.
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-o", tmp, SOURCE, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
