"""Compile the plain-C oracle into oracle/liboracle.so with gcc.

Test infrastructure: the library this builds is loaded only by the tests, the
smoke check and the benchmark's CPU-baseline leg.

Flags: no -ffast-math (subnormals and IEEE rounding must hold) and
-ffp-contract=off (no fused multiply-add, so every double op rounds once).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dtrot_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def needs_build() -> bool:
    return not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC)


def build(force: bool = False) -> str:
    if force or needs_build():
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", "-fvisibility=hidden",
               "-o", tmp, SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
