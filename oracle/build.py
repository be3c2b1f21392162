"""Compile the CPU oracle (plain C, float64) into oracle/_build/liboracle.so.

Test infrastructure: building the checker is not using it. Compiled with
-ffp-contract=off so that no fused multiply-add changes a float64 rounding,
and without any architecture flag, so x86-64 and aarch64 hosts agree.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "moe_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIBRARY = os.path.join(BUILD_DIR, "liboracle.so")


def build(force: bool = False) -> str:
    """Build the shared library if missing or older than its source; return its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    fresh = os.path.exists(LIBRARY) and os.path.getmtime(LIBRARY) >= os.path.getmtime(SOURCE)
    if fresh and not force:
        return LIBRARY
    tmp = LIBRARY + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
           "-Wall", "-o", tmp, SOURCE, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force=True))
