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
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_f64.restype = ctypes.c_double
        lib.oracle_gemm_fp8_block_scaled_rows.argtypes = [p, p, p, p, p, i64, i64, i64, i64, ctypes.c_int, p, i64]
        lib.oracle_gemm_fp8_block_scaled_rows.restype = ctypes.c_int
        lib.oracle_attention_fwd_rows.argtypes = [p, p, p, p, i64, i64, i64, i64, ctypes.c_double, ctypes.c_int,
                                                  p, i64]
        lib.oracle_attention_fwd_rows.restype = ctypes.c_int
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


# ---------------------------------------------------------------------------
# FP8 block-scaled GEMM (the TileLang-MUSA lesson, section 8.2,
# fp8_block_scaled_linear with block=128; the arithmetic is written out in
# gemm_oracle.c above oracle_gemm_fp8_block_scaled_rows).

def _as_u8(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach()
        if x.device.type != "cpu":
            raise ValueError("oracle inputs must be CPU tensors")
        if str(x.dtype).startswith("torch.float8"):
            import torch
            x = x.view(torch.uint8)
        x = x.contiguous().numpy()
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint8:
        raise TypeError(f"expected FP8 bytes (uint8), got {x.dtype}")
    return x


def _as_f32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach()
        if x.device.type != "cpu":
            raise ValueError("oracle inputs must be CPU tensors")
        x = x.contiguous().numpy()
    x = np.ascontiguousarray(x)
    if x.dtype != np.float32:
        raise TypeError(f"expected float32 scales, got {x.dtype}")
    return x


def e4m3_to_f64(codes) -> np.ndarray:
    """Decodes OCP FP8 E4M3 byte codes to float64, element by element, in C."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8).ravel()
    out = np.fromiter((lib.oracle_e4m3_to_f64(int(v)) for v in c), dtype=np.float64, count=c.size)
    return out.reshape(np.shape(codes))


def gemm_fp8_block_scaled(A, SA, W, SW, relu: bool, block: int = 128, rows=None) -> np.ndarray:
    """C = R(sum_b SA[:,b] SW[n/block,b] (A_b @ W_b^T)) as float16, by the C oracle.

    A (M,K) and W (N,K): E4M3 codes (uint8 numpy or CPU torch uint8 /
    float8_e4m3fn); SA (M, ceil(K/block)) and SW (ceil(N/block),
    ceil(K/block)): float32.  ``rows`` selects output rows as in gemm_f16.
    """
    a, w = _as_u8(A), _as_u8(W)
    sa, sw = _as_f32(SA), _as_f32(SW)
    if a.ndim != 2 or w.ndim != 2 or a.shape[1] != w.shape[1]:
        raise ValueError(f"shape mismatch: A {a.shape}, W {w.shape}")
    M, K = a.shape
    N = w.shape[0]
    KB, NB = -(-K // block), -(-N // block)
    if sa.shape != (M, KB) or sw.shape != (NB, KB):
        raise ValueError(f"scale shapes: SA {sa.shape} (want {(M, KB)}), SW {sw.shape} (want {(NB, KB)})")
    lib = _load()
    if rows is None:
        n_rows, rows_ptr = M, None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n_rows, rows_ptr = rows_arr.size, rows_arr.ctypes.data
    c = np.empty((n_rows, N), dtype=np.uint16)
    ptr = lambda x: x.ctypes.data if x.size else None
    rc = lib.oracle_gemm_fp8_block_scaled_rows(ptr(a), ptr(sa), ptr(w), ptr(sw), ptr(c), M, N, K, block,
                                               int(bool(relu)), rows_ptr, n_rows)
    if rc != 0:
        raise ValueError("oracle_gemm_fp8_block_scaled_rows rejected its arguments")
    return c.view(np.float16)


def e8m0_to_f32(codes) -> np.ndarray:
    """Decodes E8M0 scale bytes (the OCP microscaling formats' scale type: an
    8-bit biased exponent and nothing else) to float32: code c < 255 is
    2^(c - 127), code 255 is NaN.  Every value is exact in float32 (2^-127 is a
    subnormal)."""
    c = np.asarray(codes, dtype=np.int64)
    out = np.ldexp(np.float32(1.0), (c - 127).astype(np.int32)).astype(np.float32)
    return np.where(c == 255, np.float32(np.nan), out).astype(np.float32)


def gemm_mxfp8_block_scaled(A, SA, W, SW, relu: bool, rows=None) -> np.ndarray:
    """The FP8 block-scaled GEMM with power-of-two scales given as E8M0 bytes:
    C = R(sum_b 2^(SA[i,b]-127) 2^(SW[n/128,b]-127) (A_b @ W_b^T)) as float16.
    The scales are decoded exactly and the product is the one of
    gemm_fp8_block_scaled (blocks of 128)."""
    sa, sw = _as_u8(SA), _as_u8(SW)
    return gemm_fp8_block_scaled(A, e8m0_to_f32(sa), W, e8m0_to_f32(sw), relu=relu, block=128, rows=rows)


# ---------------------------------------------------------------------------
# Attention forward (the FlashAttention skeleton of the TileLang-MUSA lesson,
# section 5; the plain definition is written out in gemm_oracle.c above
# oracle_attention_fwd_rows).

def attention_fwd(Q, K, V, sm_scale: float, causal: bool, rows=None) -> np.ndarray:
    """O = softmax(sm_scale Q K^T [causal mask]) V per (batch, head), fp16 out.

    Q, K, V: (batch, heads, seq, dim) float16 (numpy, uint16 bits or CPU
    torch).  Without ``rows`` returns O (batch, heads, seq, dim); with
    ``rows`` (flat indices (b*heads + h)*seq + i) returns those rows stacked,
    shape (len(rows), dim).
    """
    q, k, v = _as_f16_bits(Q), _as_f16_bits(K), _as_f16_bits(V)
    if q.ndim != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError(f"Q, K, V must share one (batch, heads, seq, dim) shape: {q.shape} {k.shape} {v.shape}")
    B, H, S, D = q.shape
    lib = _load()
    if rows is None:
        n_rows, rows_ptr = B * H * S, None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n_rows, rows_ptr = rows_arr.size, rows_arr.ctypes.data
    o = np.empty((n_rows, D), dtype=np.uint16)
    ptr = lambda x: x.ctypes.data if x.size else None
    rc = lib.oracle_attention_fwd_rows(ptr(q), ptr(k), ptr(v), ptr(o), B, H, S, D, float(sm_scale),
                                       int(bool(causal)), rows_ptr, n_rows)
    if rc != 0:
        raise ValueError("oracle_attention_fwd_rows rejected its arguments")
    o = o.view(np.float16)
    return o.reshape(B, H, S, D) if rows is None else o
