"""Compile the float64 oracle (test infrastructure) into oracle/liboracle.so.

Building the checker is not using it: ``__graft_entry__.build()`` calls
this so the tests find the library, but only the tests, the smoke check and
the benchmark's CPU-baseline leg load it.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    # -ffp-contract=off: no fused multiply-add, so every product and sum is
    # rounded as written; -O2 without -ffast-math keeps IEEE semantics.
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-pthread", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
