"""Build the CPU oracle's shared library (TEST INFRASTRUCTURE ONLY).

The oracle is compiled with ``-ffp-contract=off -fno-fast-math`` so that no
``a*b + c`` is fused into an FMA: the FP32 epilogue on the pages is built with
FMA contraction turned off ("Fuse Beam's TP all-reduce with its sandwich
norms", section "Details", "Build" bullet), and GCC on aarch64 contracts by
default.  The output goes to ``oracle/_build/liboracle.so`` (git-ignored).
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "beamnorm_oracle.c")
HDR = os.path.join(HERE, "beamnorm_oracle.h")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
          "-Wall", "-Wextra", "-Werror"]


def build(force: bool = False) -> str:
    """Compile the oracle if the library is missing or older than its sources."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB):
        newest = max(os.path.getmtime(SRC), os.path.getmtime(HDR), os.path.getmtime(__file__))
        if os.path.getmtime(LIB) >= newest:
            return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, "-shared", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
