"""Build the CPU oracle shared library (test infrastructure only).

The oracle is plain C11, single-threaded, compiled without fast-math and with
floating-point contraction off, so that each f32 operation in the source is the
IEEE-754 operation that runs.  Building it is not using it: the package build
compiles it alongside the CUDA library so that the tests find it ready.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "rz_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liborc.so")
LIB_OMP = os.path.join(OUT_DIR, "liborc_omp.so")

CFLAGS = ["-std=c11", "-O2", "-Wall", "-Wextra", "-ffp-contract=off",
          "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False, openmp: bool = False) -> str:
    """Compile rz_oracle.c into _build/liborc.so (single-threaded), or with
    openmp=True into _build/liborc_omp.so: the same source with its independent
    output rows split over all host cores (the all-core CPU baseline; every row is
    still summed in the same order, so results are identical)."""
    os.makedirs(OUT_DIR, exist_ok=True)
    lib = LIB_OMP if openmp else LIB
    deps = [SRC, os.path.join(HERE, "rz_oracle.h")]
    if not force and os.path.exists(lib):
        if os.path.getmtime(lib) >= max(os.path.getmtime(p) for p in deps):
            return lib
    tmp = lib + ".tmp.%d" % os.getpid()
    cmd = ["gcc", *CFLAGS, *(["-fopenmp"] if openmp else []), "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
    print(build(force="--force" in sys.argv, openmp=True))
