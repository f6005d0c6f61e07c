"""Compile the C oracle into ``oracle/_build/libcsa_oracle.so`` with gcc.

Test infrastructure only (see ``oracle/__init__.py``). OpenMP is used when
the compiler supports it; otherwise the oracle runs single-threaded.
"""

from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csa_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libcsa_oracle.so")


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra", SRC, "-o", tmp, "-lm"]
    for extra in (["-fopenmp"], []):
        cmd = base[:2] + extra + base[2:]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode == 0:
            if verbose:
                print(" ".join(cmd))
            os.replace(tmp, LIB)
            return LIB
    raise RuntimeError("oracle build failed:\n" + res.stderr)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
