"""Compile the CPU oracle (plain C, fp64) into oracle/_build/libmlaoracle.so.

TEST INFRASTRUCTURE: the oracle is built so that tests, the smoke check and
the benchmark's CPU baseline can run it; the product path never loads it.
Portable flags only (the same source builds on x86_64 and aarch64).
"""

from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "mla_verify_oracle.c")
SRCS = [SRC, os.path.join(HERE, "next_rows_oracle.c")]
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libmlaoracle.so")


def build(force: bool = False, verbose: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and all(os.path.getmtime(LIB) >= os.path.getmtime(f) for f in SRCS)):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", *SRCS, "-o", tmp, "-lm"]
    cmd = base[:1] + ["-fopenmp"] + base[1:]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        if verbose:
            print("oracle: OpenMP build failed, building single-threaded:\n" + r.stderr,
                  file=sys.stderr)
        r = subprocess.run(base, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
