"""Compile the CPU oracle (sgemm_oracle.c) into liboracle.so with gcc.

Plain C11, -O2, no fast-math and no floating-point contraction, so the
fp64 sums round exactly as written; the same flags work on x86-64 and
aarch64.  Rebuilds when the source is newer than the library.
"""
from __future__ import annotations

import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "sgemm_oracle.c")
LIB = os.path.join(_HERE, "liboracle.so")
CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread"]


def build_oracle(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cc = os.environ.get("CC", "gcc")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *CFLAGS, SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))
