"""Compile the CPU oracle (``oracle.c``) into ``oracle/_build/liboracle.so``.

Test infrastructure: the oracle is built so that the tests, the smoke check and the
benchmark's CPU baseline can call it. ``-ffp-contract=off`` keeps every product and
sum a separately rounded operation, as the oracle's precision argument requires.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")

_BASE = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source; return its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    try:
        subprocess.run(_BASE + ["-fopenmp", SRC, "-o", tmp, "-lm"], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        # OpenMP only spreads independent work (pairs, blocks of tokens) over cores.
        subprocess.run(_BASE + [SRC, "-o", tmp, "-lm"], check=True, capture_output=True, text=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
