"""Compile the fp64 selective-scan oracle (test infrastructure) into a shared object.

The oracle is plain C; it is built with gcc, with OpenMP over (batch, channel) rows
when the compiler supports it and without it otherwise.  Only the test suite, the
smoke check and the benchmark's CPU-baseline leg load the result.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "selscan_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False, verbose: bool = False) -> str:
    """Build ``liboracle.so`` next to its source when missing or stale; return its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", SRC, "-o", tmp, "-lm"]
    errors = []
    for extra in (["-fopenmp"], []):
        cmd = base[:2] + extra + base[2:]
        proc = subprocess.run(cmd, capture_output=True, text=True)
        if proc.returncode == 0:
            os.replace(tmp, LIB)
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            return LIB
        errors.append(f"{' '.join(cmd)}\n{proc.stderr}")
    raise RuntimeError("oracle build failed:\n" + "\n".join(errors))


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
