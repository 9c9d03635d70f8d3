"""GB300-native fused fp16 GEMM + ReLU: C = ReLU(A @ B) (or A @ B).

The product is the C-ABI library ``libgemm_f16.so`` (declared in
``include/gemm_f16.h``) with hand-written sm_103a kernels behind it;
``gemm_f16`` (this package's module of the same name) is the thin ctypes
binding over it.  ``inputs`` holds the seeded synthetic operand generators.

The binding is imported lazily so that ``inputs`` can be used on machines
without the built library.
"""
from __future__ import annotations

__all__ = ["gemm_f16", "inputs"]


def __getattr__(name):
    if name in ("gemm_f16", "inputs", "build"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
