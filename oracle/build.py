"""Builds the oracle shared library (test infrastructure) with g++.

`-ffp-contract=off` keeps every written fp32 operation a separate rounding
(GCC fuses a*b+c by default on some targets, AArch64 among them).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.cpp")
LIB = os.path.join(HERE, "liboracle.so")


FLAGS = ["-std=c++17", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra"]


def compile_oracle(src: str, out: str) -> str:
    subprocess.check_call(["g++", *FLAGS, "-o", out, src])
    return out


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    compile_oracle(SRC, tmp)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
