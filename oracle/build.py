"""Build the CPU oracle shared library (test infrastructure only).

Compiles ``qmm_oracle.c`` with plain ``-O2`` (no fast-math, no FMA contraction,
so every fp32 step rounds as written) and OpenMP over output rows when the
compiler supports it.  The result lands in ``oracle/_build/`` and is never
linked into the product library.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "qmm_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")

_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-fno-strict-aliasing"]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the oracle if the shared library is missing or stale; return its path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    cc = os.environ.get("CC", "gcc")
    tmp = LIB + f".tmp{os.getpid()}"
    for omp in (["-fopenmp"], []):
        cmd = [cc, *_FLAGS, *omp, SRC, "-o", tmp, "-lm"]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(tmp, LIB)
            return LIB
    raise RuntimeError(f"oracle build failed:\n{r.stderr}")


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
