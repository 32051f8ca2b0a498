"""Builds the CPU oracle's shared library (test infrastructure only).

The oracle is plain C compiled without fast-math or floating-point
contraction, so that every binary32 operation in it is one IEEE-754
operation rounded to nearest-even.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-pthread", "-std=c11", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compiles oracle.c into liboracle.so next to it; returns the path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, SRC, "-lm"])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
