"""Compile the CPU oracle (tl_oracle.c) into oracle/libtl_oracle.so.

Test infrastructure: building the checker is not using it.  Plain gcc, -O2,
no fast-math, no FMA contraction, no intrinsics.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "tl_oracle.c")
LIB = os.path.join(HERE, "libtl_oracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fno-tree-vectorize", "-pthread", "-shared", "-fPIC", SRC,
           "-o", LIB + ".tmp", "-lm"]
    subprocess.check_call(cmd)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
