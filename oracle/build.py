"""Compile the CPU oracle (plain C, fp64) into oracle/_build/libspec_oracle.so.

Test infrastructure: built by the package build step so that the tests, the
smoke check and the benchmark's CPU baseline can load it.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "spec_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libspec_oracle.so")


def compile_oracle(src: str = SRC, out: str = LIB, extra=()) -> str:
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", *extra, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    return compile_oracle()


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
