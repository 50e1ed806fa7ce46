"""Build the oracle's shared library with the host C compiler.

Plain C99 + OpenMP, no fast math and no FMA contraction, so every fp32
operation in ``oracle.c`` is a single IEEE-rounded operation on x86-64 and
aarch64 alike.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB_PATH = os.path.join(HERE, "liboracle.so")


def build(verbose: bool = False) -> str:
    cc = os.environ.get("CC", "gcc")
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [cc, "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wno-unused-function",
           SRC, "-o", tmp, "-lm"]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(verbose=True))
