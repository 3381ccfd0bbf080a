"""Compile the CPU oracle (test infrastructure) into oracle/_build/.

gcc, -O2, strict IEEE fp64 (no fast-math, no FMA contraction), OpenMP when
the compiler has it.  Rebuilt when the source is newer or the library was
made on another machine (a stamp file records it).  Prints one line saying
what it did.
"""
from __future__ import annotations

import os
import platform
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "msa_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libmsa_oracle.so")


def build(force: bool = False, verbose: bool = False) -> str:
    stamp_file = os.path.join(OUT_DIR, "stamp.txt")
    try:
        same_machine = open(stamp_file).read().strip() == platform.machine()
    except OSError:
        same_machine = False
    if not force and same_machine and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        print(f"oracle build ({platform.machine()}): up to date: {LIB}")
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + f".{os.getpid()}.tmp"
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC", SRC, "-o", tmp, "-lm"]
    for extra in (["-fopenmp"], []):
        cmd = base[:1] + extra + base[1:]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode == 0:
            os.replace(tmp, LIB)
            with open(stamp_file, "w") as f:
                f.write(platform.machine() + "\n")
            if verbose:
                print(" ".join(cmd))
            print(f"oracle build ({platform.machine()}): compiled{' with OpenMP' if extra else ''}: {LIB}")
            return LIB
    raise RuntimeError("oracle build failed:\n" + res.stderr)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
