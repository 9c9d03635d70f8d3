"""CPU oracle for C = ReLU(A @ B) on fp16 operands -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg import this package.  The product library never does, and the
oracle imports nothing from the product package: the two share no code.

The arithmetic lives in ``gemm_oracle.c`` (plain C, fp64 accumulation, IEEE
round-to-nearest-even written out by hand).  This module only marshals numpy
arrays into it.  What it follows, on "Writing High-Performance Kernels in
TileLang, from GEMM to MLA" (atlascloud.ai), section "Let's write a GEMM":
C = ReLU(A @ B) for row-major A (M,K), B (K,N), C (M,N) in float16, with the
accumulator in float and the ReLU applied to the accumulator before the
write-back cast.

Every function here is pinned by ``tests/test_oracle_pins.py`` against facts
that do not come from the oracle itself: numpy's binary16 conversions on all
65,536 bit patterns and on ties, closed forms (identity, permutation, all
negative products), an int64 brute-force matmul on small integers and the
hand-derived cases in ``tests/golden/``.
"""
from __future__ import annotations

import ctypes
import os
import time

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        lib.oracle_f64_to_f16.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_f16.restype = ctypes.c_uint16
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        lib.oracle_gemm_f16_rows.argtypes = [p, p, p, i64, i64, i64, ctypes.c_int, p, i64]
        lib.oracle_gemm_f16_rows.restype = ctypes.c_int
        lib.oracle_relu_backward.argtypes = [p, p, p, i64]
        lib.oracle_relu_backward.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _as_f16_bits(x) -> np.ndarray:
    """Accepts a float16 numpy array, a uint16 bit array or a CPU torch tensor."""
    if hasattr(x, "detach"):  # torch tensor, CPU only (the oracle never touches a GPU)
        x = x.detach()
        if x.device.type != "cpu":
            raise ValueError("oracle inputs must be CPU tensors")
        x = x.contiguous().numpy()
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        return x.view(np.uint16)
    if x.dtype == np.uint16:
        return x
    raise TypeError(f"expected float16 or uint16 bits, got {x.dtype}")


def f16_to_f64(bits) -> np.ndarray:
    """Decodes binary16 bit patterns to float64, element by element, in C."""
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16).ravel()
    out = np.fromiter((lib.oracle_f16_to_f64(int(v)) for v in b), dtype=np.float64, count=b.size)
    return out.reshape(np.shape(bits))


def f64_to_f16_bits(values) -> np.ndarray:
    """Rounds float64 values to binary16 (nearest, ties to even); returns uint16 bits."""
    lib = _load()
    v = np.asarray(values, dtype=np.float64).ravel()
    out = np.fromiter((lib.oracle_f64_to_f16(float(x)) for x in v), dtype=np.uint16, count=v.size)
    return out.reshape(np.shape(values))


def gemm_f16(A, B, relu: bool, rows=None) -> np.ndarray:
    """C = R(A @ B) as float16, computed by the C oracle.

    A: (M,K) and B: (K,N) float16 (numpy, uint16 bits or CPU torch).  With
    ``rows`` (a sequence of row indices) only those output rows are computed
    and returned, stacked in the given order, shape (len(rows), N).
    """
    a = _as_f16_bits(A)
    b = _as_f16_bits(B)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[0]:
        raise ValueError(f"shape mismatch: A {a.shape}, B {b.shape}")
    M, K = a.shape
    N = b.shape[1]
    lib = _load()
    if rows is None:
        n_rows = M
        rows_arr = None
        rows_ptr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n_rows = rows_arr.size
        rows_ptr = rows_arr.ctypes.data
    c = np.empty((n_rows, N), dtype=np.uint16)
    rc = lib.oracle_gemm_f16_rows(
        a.ctypes.data if a.size else None, b.ctypes.data if b.size else None,
        c.ctypes.data if c.size else None, M, N, K, int(bool(relu)), rows_ptr, n_rows)
    if rc != 0:
        raise ValueError("oracle_gemm_f16_rows rejected its arguments")
    return c.view(np.float16)


def num_threads() -> int:
    """Threads an OpenMP region of the oracle uses (OMP_NUM_THREADS, else all cores)."""
    return int(_load().oracle_num_threads())


def time_rows(A, B, relu: bool, rows) -> tuple[np.ndarray, float]:
    """Runs :func:`gemm_f16` on the given rows and returns (C_rows, seconds)."""
    t0 = time.perf_counter()
    c = gemm_f16(A, B, relu, rows=rows)
    return c, time.perf_counter() - t0


def relu_backward(dC, C) -> np.ndarray:
    """dZ = dC where C > 0 else +0 (the ReLU gradient), float16, by the C oracle."""
    g = _as_f16_bits(dC)
    c = _as_f16_bits(C)
    if g.shape != c.shape:
        raise ValueError(f"shape mismatch: dC {g.shape}, C {c.shape}")
    out = np.empty(g.shape, dtype=np.uint16)
    if g.size:
        _load().oracle_relu_backward(g.ctypes.data, c.ctypes.data, out.ctypes.data, g.size)
    return out.view(np.float16)


def gemm_f16_t(A, B, relu: bool, transa: bool = False, transb: bool = False, rows=None) -> np.ndarray:
    """C = R(op(A) @ op(B)): op(X) is X or its transpose (numpy transposes the
    stored matrix; the product itself is the oracle's gemm_f16)."""
    a = _as_f16_bits(A)
    b = _as_f16_bits(B)
    if transa:
        a = np.ascontiguousarray(a.T)
    if transb:
        b = np.ascontiguousarray(b.T)
    return gemm_f16(a, b, relu, rows=rows)
