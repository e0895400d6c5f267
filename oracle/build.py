"""Compile the CPU oracle (oracle.c) into liboracle.so with gcc.

Test infrastructure only: the oracle is the slow fp64 reference the GPU path is checked
against.  The build is plain gcc + OpenMP, no CUDA, and writes the library next to this
file.  ``-ffp-contract=off`` keeps every multiply and add a separately rounded operation,
as written in the C source.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def needs_build() -> bool:
    return (not os.path.exists(LIB)) or os.path.getmtime(LIB) < os.path.getmtime(SRC)


def build(force: bool = False) -> str:
    if force or needs_build():
        tmp = LIB + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
               SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
