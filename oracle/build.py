"""Builds the CPU oracle (``gemm_oracle.c``) into ``oracle/liboracle_gemm.so``.

TEST INFRASTRUCTURE: the oracle is the independent CPU reference used by the
tests, the smoke check and the bench's CPU-baseline leg.  Building it is not
using it; ``__graft_entry__.build()`` calls :func:`build` so that the checker
exists wherever the GPU library is built.

Plain gcc, no CUDA, no vector intrinsics: the same source builds on x86_64 and
aarch64.  ``-ffp-contract=off`` keeps every ``acc += a * b`` a separately
rounded multiply and add (exactly what the source says; no fused multiply-add).
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gemm_oracle.c")
LIB = os.path.join(HERE, "liboracle_gemm.so")


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles the oracle if the shared library is missing or older than its source."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [
        os.environ.get("CC", "gcc"), "-O2", "-fopenmp", "-ffp-contract=off",
        "-fno-fast-math", "-shared", "-fPIC", "-Wall", "-Wextra",
        "-o", tmp, SRC, "-lm",
    ]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
