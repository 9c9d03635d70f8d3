"""torch.autograd wrapper around the library's kernels (training use).

The TileLang-MUSA lesson (7yue.com, section 6, "wrapping a TileLang kernel for
PyTorch") wraps its GEMM kernel in a ``torch.autograd.Function`` whose forward
calls the kernel and whose backward returns ``dA = dC @ B.T`` and
``dB = A.T @ dC``.  Here every step runs in this library's sm_103a kernels:

* forward   C = R(A @ B)                         gemm_f16_tx (NN)
* ReLU      dZ = dC where C > 0, else +0         gemm_f16_relu_backward (only with ReLU)
* dA        dZ @ B^T   (B stored (K,N))          gemm_f16_tx with transb = 1 (NT)
* dB        A^T @ dZ   (A stored (M,K))          gemm_f16_tx with transa = 1 (TN)

Operands and gradients are float16 (the kernels accumulate in fp32).  No step
falls back to torch arithmetic; a missing library raises LibraryNotBuilt.
"""
from __future__ import annotations

import torch

from . import gemm_f16 as _g


class GemmF16Function(torch.autograd.Function):
    """C = ReLU(A @ B) (relu=True) or A @ B, with the backward pair above."""

    @staticmethod
    def forward(ctx, A: torch.Tensor, B: torch.Tensor, relu: bool = True):
        A = A.contiguous()
        B = B.contiguous()
        C = _g.gemm_f16_t(A, B, relu=relu)
        ctx.relu = bool(relu)
        ctx.save_for_backward(A, B, C if relu else None)
        return C

    @staticmethod
    def backward(ctx, dC: torch.Tensor):
        A, B, C = ctx.saved_tensors
        dC = dC.contiguous()
        if dC.dtype != torch.float16:
            dC = dC.half()
        dZ = _g.relu_backward(dC, C) if ctx.relu else dC
        dA = dB = None
        if ctx.needs_input_grad[0]:
            dA = _g.gemm_f16_t(dZ, B, transb=True, relu=False)     # (M,N) @ (N,K)
        if ctx.needs_input_grad[1]:
            dB = _g.gemm_f16_t(A, dZ, transa=True, relu=False)     # (K,M) @ (M,N)
        return dA, dB, None


def gemm_relu(A: torch.Tensor, B: torch.Tensor) -> torch.Tensor:
    """Differentiable C = ReLU(A @ B) on fp16 CUDA tensors."""
    return GemmF16Function.apply(A, B, True)


def gemm(A: torch.Tensor, B: torch.Tensor) -> torch.Tensor:
    """Differentiable C = A @ B on fp16 CUDA tensors (the lesson's TLGemm)."""
    return GemmF16Function.apply(A, B, False)
