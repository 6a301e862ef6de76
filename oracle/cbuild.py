"""Builds the C++ oracle (moe_oracle.cpp) into oracle/lib/liboracle_moe.so.

TEST INFRASTRUCTURE: the library is the checker the tests, the smoke check
and the benchmark's CPU legs run; the CUDA library never links or loads it.
Plain g++ (C++17, OpenMP), no machine-specific flags, and -ffp-contract=off so
that no multiply-add is fused and results are the same on every host.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.cpp")
LIBDIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIBDIR, "liboracle_moe.so")
FLAGS = ["-O3", "-std=c++17", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off",
         "-Wall", "-Wextra"]


def compiler() -> str:
    for cand in (os.environ.get("CXX"), shutil.which("g++"), "/usr/bin/g++"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("g++ not found")


def build(force: bool = False) -> str:
    """Compile the oracle library if its source or flags changed; returns its path."""
    os.makedirs(LIBDIR, exist_ok=True)
    with open(SRC, "rb") as f:
        stamp = hashlib.sha256(f.read() + " ".join(FLAGS).encode()).hexdigest()
    stamp_file = os.path.join(LIBDIR, "stamp")
    if not force and os.path.exists(LIB) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read() == stamp:
                return LIB
    tmp = LIB + ".tmp"
    r = subprocess.run([compiler(), *FLAGS, SRC, "-o", tmp], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"oracle build failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv[1:]))
