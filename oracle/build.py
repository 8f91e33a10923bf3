"""Compile the reference oracle (fq_oracle.cpp) into oracle/_build/libfq_oracle.so.

Test infrastructure: the library this builds is loaded only by the test suite, the package smoke
check and the benchmark's CPU-baseline leg. Plain g++, no CUDA.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fq_oracle.cpp")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libfq_oracle.so")

# -ffp-contract=off: a*b+c stays two roundings, like the separate fp32 tensor ops it restates.
CXXFLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source; return its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["g++", *CXXFLAGS, SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)  # atomic: concurrent builders never see a half-written library
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
