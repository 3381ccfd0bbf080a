"""Compile the CPU oracle (test infrastructure) into oracle/_build/.

gcc, -O2, strict IEEE fp64 (no fast-math, no FMA contraction), OpenMP when
the compiler has it.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "msa_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libmsa_oracle.so")


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + f".{os.getpid()}.tmp"
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC", SRC, "-o", tmp, "-lm"]
    for extra in (["-fopenmp"], []):
        cmd = base[:1] + extra + base[1:]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode == 0:
            os.replace(tmp, LIB)
            if verbose:
                print(" ".join(cmd))
            return LIB
    raise RuntimeError("oracle build failed:\n" + res.stderr)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
