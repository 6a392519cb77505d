"""Compile the CPU oracle (``oracle.c``) into ``oracle/_build/liboracle.so``.

Test infrastructure: the library is built with plain gcc, fp-contraction
off and no fast-math, so every fp64 operation is the one written in the
source.  OpenMP is used when the compiler offers it (only to spread output
rows over host threads; each output is still one sequential sum).
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


def _compile(extra: list[str]) -> subprocess.CompletedProcess:
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", *extra, SRC, "-o", LIB + ".tmp", "-lm"]
    return subprocess.run(cmd, capture_output=True, text=True)


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    res = _compile(["-fopenmp"])
    if res.returncode != 0:  # no OpenMP runtime: single-threaded oracle
        res = _compile([])
    if res.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + res.stderr)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
