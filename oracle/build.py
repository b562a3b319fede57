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

FLAGS = ["-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and all(os.path.getmtime(LIB) >= os.path.getmtime(s) for s in SRCS)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["g++", *FLAGS, *SRCS, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
