"""Compile the CPU oracle into oracle/liboracle.so.

TEST INFRASTRUCTURE: the oracle is only loaded by tests/, by
__graft_entry__.smoke() and by bench.py's CPU-baseline and reference legs.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "nvfp4_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

# IEEE binary32/64 evaluation exactly as written: no FMA contraction, no
# fast-math reassociation, no flush-to-zero.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
          "-ffp-contract=off", "-fno-fast-math", "-fno-finite-math-only"]


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp"
    subprocess.check_call(["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
