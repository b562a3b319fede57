"""Compile the CPU oracle (oracle.cpp, project.cpp) into oracle/_build/liboracle.so.

Test infrastructure: the oracle checks the CUDA library and is never called
by it.  Plain g++, no contraction of a*b+c into FMA (-ffp-contract=off), so
every float expression rounds as written on x86 and on Arm alike.
"""

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRCS = [os.path.join(HERE, "oracle.cpp"), os.path.join(HERE, "project.cpp")]
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")
# the same sources with OpenMP: pixels on every host core (timing only; the
# tests load the single-threaded LIB)
LIB_OMP = os.path.join(OUT_DIR, "liboracle_omp.so")

FLAGS = ["-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def _build_one(out, extra, force):
    if (not force and os.path.exists(out)
            and all(os.path.getmtime(out) >= os.path.getmtime(s) for s in SRCS)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["g++", *FLAGS, *extra, *SRCS, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False, omp: bool = False) -> str:
    """Builds both libraries; returns the path of the one asked for."""
    os.makedirs(OUT_DIR, exist_ok=True)
    _build_one(LIB, [], force)
    _build_one(LIB_OMP, ["-fopenmp"], force)
    return LIB_OMP if omp else LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
