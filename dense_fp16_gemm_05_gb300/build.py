"""Builds the CUDA library ``libgemm_f16.so`` in-tree with nvcc for sm_103a.

Translation units: ``csrc/gemm_f16.cu`` (the C ABI) and ``csrc/gemm_cfg_<id>.cu``
(the kernel instances of each configuration), compiled in parallel with one
``-gencode`` (``arch=compute_103a,code=sm_103a``) and linked with the CUDA
runtime linked statically, so the library loads on machines without a GPU
driver (the symbol-export test runs there).  The build is skipped when the
library is newer than every source.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libgemm_f16.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo", "-O3", "-std=c++17",
    "-shared", "-Xcompiler", "-fPIC",
    "-cudart", "static",
]


def _sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(CSRC, "*.inc")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _translation_units() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None) -> str:
    """Compiles the library if it is missing or stale; returns its path.

    Each translation unit (the C ABI and one per kernel configuration) is
    compiled to an object in parallel, then the objects are linked into one
    shared library.
    """
    if not force and os.path.exists(LIB):
        lib_t = os.path.getmtime(LIB)
        if all(os.path.getmtime(s) <= lib_t for s in _sources()):
            return LIB
    import concurrent.futures
    import tempfile
    tmpdir = tempfile.mkdtemp(prefix="gemm_f16_build")
    compile_flags = [f for f in NVCC_FLAGS if f not in ("-shared", "-cudart", "static")]
    units = _translation_units()

    def compile_one(src):
        obj = os.path.join(tmpdir, os.path.basename(src) + ".o")
        cmd = [nvcc(), *compile_flags, *(extra_flags or []), "-I", INCLUDE, "-c", "-o", obj, src]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        subprocess.run(cmd, check=True)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=min(len(units), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, units))
    tmp = LIB + f".tmp{os.getpid()}"
    link = [nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-cudart", "static", "-o", tmp, *objs]
    if verbose:
        print(" ".join(link), file=sys.stderr)
    subprocess.run(link, check=True)
    os.replace(tmp, LIB)
    for o in objs:
        os.unlink(o)
    os.rmdir(tmpdir)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
