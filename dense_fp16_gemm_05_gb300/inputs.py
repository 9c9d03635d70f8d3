"""Seeded synthetic inputs for the fp16 GEMM + ReLU workloads.

This module holds no GEMM arithmetic: it only draws operands.  The same bits
feed the CUDA path and the CPU oracle (tests copy the CPU tensors to the
device), so neither side generates its own data.

Recipe (the pages draw both operands with ``torch.randn`` in float16 and check
1024^3; the larger configurations scale by 1/sqrt(K) so that |C| stays O(1)):

* ``normal``: float32 N(0,1) from ``torch.Generator().manual_seed(seed)``,
  optionally multiplied by float32(1/sqrt(K)), rounded to float16 by
  ``Tensor.half()`` (round to nearest even; subnormals kept).
* ``integer``: integers drawn uniformly from {-4, ..., 4} with
  ``torch.randint``, converted to float16 (exact).

A is drawn first, then B, from one generator.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    """One GEMM problem: C = R(A @ B), A (M,K), B (K,N), all float16 row-major."""
    name: str
    M: int
    N: int
    K: int
    relu: bool
    values: str          # "normal", "normal_scaled" (N(0,1)/sqrt(K)) or "integer"
    seed: int

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


def draw(M: int, N: int, K: int, values: str, seed: int) -> tuple[torch.Tensor, torch.Tensor]:
    """Returns CPU float16 tensors A (M,K) and B (K,N) drawn from ``seed``."""
    g = torch.Generator().manual_seed(int(seed))
    if values in ("normal", "normal_scaled"):
        a = torch.randn(M, K, generator=g, dtype=torch.float32)
        b = torch.randn(K, N, generator=g, dtype=torch.float32)
        if values == "normal_scaled" and K > 0:
            s = torch.tensor(1.0 / math.sqrt(K), dtype=torch.float32)
            a = a * s
            b = b * s
        return a.half(), b.half()
    if values == "integer":
        a = torch.randint(-4, 5, (M, K), generator=g, dtype=torch.int32)
        b = torch.randint(-4, 5, (K, N), generator=g, dtype=torch.int32)
        return a.half(), b.half()
    raise ValueError(f"unknown value recipe {values!r}")


def draw_workload(w: Workload) -> tuple[torch.Tensor, torch.Tensor]:
    return draw(w.M, w.N, w.K, w.values, w.seed)


def draw_on_device(M: int, N: int, K: int, values: str, seed: int,
                   device: torch.device) -> tuple[torch.Tensor, torch.Tensor]:
    """The ``normal`` / ``normal_scaled`` recipe drawn by a seeded generator on
    ``device`` (same distribution as ``draw``, other bits): for timing runs
    whose operands are too large to draw quickly on the host and that compare
    nothing against the oracle."""
    if values not in ("normal", "normal_scaled"):
        raise ValueError(f"device drawing supports the normal recipes, not {values!r}")
    g = torch.Generator(device=device).manual_seed(int(seed))
    a = torch.randn(M, K, generator=g, dtype=torch.float32, device=device)
    b = torch.randn(K, N, generator=g, dtype=torch.float32, device=device)
    if values == "normal_scaled" and K > 0:
        s = torch.tensor(1.0 / math.sqrt(K), dtype=torch.float32, device=device)
        a = a * s
        b = b * s
    return a.half(), b.half()


# The five configurations of the benchmark description, with their seeds.
WORKLOADS: dict[str, Workload] = {
    "relu_1024": Workload("relu_1024", 1024, 1024, 1024, True, "normal", 1),
    "relu_ragged_1000": Workload("relu_ragged_1000", 1000, 1000, 1000, True, "normal", 2),
    "int_64": Workload("int_64", 64, 64, 64, True, "integer", 3),
    "plain_4096": Workload("plain_4096", 4096, 4096, 4096, False, "normal", 4),
    "relu_8192": Workload("relu_8192", 8192, 8192, 8192, True, "normal_scaled", 5),
}
for _n in (512, 1024, 2048, 4096, 8192, 16384):
    WORKLOADS[f"sweep_{_n}"] = Workload(f"sweep_{_n}", _n, _n, _n, True, "normal_scaled",
                                        100 + int(math.log2(_n)))


# ---------------------------------------------------------------------------
# FP8 block-scaled operands.  The TileLang-MUSA lesson (section 8.2) feeds
# fp8_block_scaled_linear an FP8 weight with per-128-block scales; nothing on
# the pages says how the operands were quantized, so the inputs are made the
# usual way (this is input synthesis, not the GEMM): each block's scale is its
# largest magnitude over 448 (the largest finite E4M3 value), and the block is
# divided by its scale and rounded to E4M3 by torch's float8_e4m3fn
# conversion.  A gets one scale per row per 128 K elements, W (N,K) one per
# 128 x 128 block.  Scales are float32.

FP8_BLOCK = 128


@dataclass(frozen=True)
class Fp8Workload:
    """C = R(sum_b SA[:,b] SW[n/128,b] A_b W_b^T): A (M,K), W (N,K) E4M3."""
    name: str
    M: int
    N: int
    K: int
    relu: bool
    values: str          # "normal" (N(0,1) quantized per block) or "integer" (exact, power-of-two scales)
    seed: int

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


def _quantize_blocks(x: torch.Tensor, rows_per_block: int, block: int) -> tuple[torch.Tensor, torch.Tensor]:
    """x (R, K) float32 -> (E4M3 codes as uint8 (R, K), float32 scales
    (ceil(R/rows_per_block), ceil(K/block)))."""
    R, K = x.shape
    RB, KB = -(-R // rows_per_block), -(-K // block)
    pad = torch.zeros(RB * rows_per_block, KB * block, dtype=torch.float32)
    pad[:R, :K] = x
    blocks = pad.view(RB, rows_per_block, KB, block)
    amax = blocks.abs().amax(dim=(1, 3))
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax)).to(torch.float32)
    q = (blocks / scale[:, None, :, None]).clamp(-448.0, 448.0)
    codes = q.reshape(RB * rows_per_block, KB * block)[:R, :K].contiguous().to(torch.float8_e4m3fn)
    return codes.view(torch.uint8), scale


def draw_fp8_block_scaled(M: int, N: int, K: int, values: str, seed: int, block: int = FP8_BLOCK):
    """CPU tensors (A codes (M,K) uint8, SA (M,KB) f32, W codes (N,K) uint8,
    SW (NB,KB) f32) drawn from ``seed``."""
    g = torch.Generator().manual_seed(int(seed))
    KB, NB = -(-K // block), -(-N // block)
    if values == "normal":
        a = torch.randn(M, K, generator=g, dtype=torch.float32)
        w = torch.randn(N, K, generator=g, dtype=torch.float32) * (1.0 / math.sqrt(max(K, 1)))
        A, SA = _quantize_blocks(a, 1, block)
        W, SW = _quantize_blocks(w, block, block)
        return A, SA, W, SW
    if values == "integer":
        a = torch.randint(-4, 5, (M, K), generator=g, dtype=torch.int32).to(torch.float32)
        w = torch.randint(-4, 5, (N, K), generator=g, dtype=torch.int32).to(torch.float32)
        ea = torch.randint(-3, 4, (M, KB), generator=g, dtype=torch.int32)
        ew = torch.randint(-3, 4, (NB, KB), generator=g, dtype=torch.int32)
        SA = torch.ldexp(torch.ones(M, KB), ea.to(torch.float32)).to(torch.float32)
        SW = torch.ldexp(torch.ones(NB, KB), ew.to(torch.float32)).to(torch.float32)
        A = a.to(torch.float8_e4m3fn).view(torch.uint8)
        W = w.to(torch.float8_e4m3fn).view(torch.uint8)
        return A, SA, W, SW
    raise ValueError(f"unknown value recipe {values!r}")


def _quantize_blocks_pow2(x: torch.Tensor, rows_per_block: int, block: int) -> tuple[torch.Tensor, torch.Tensor]:
    """As _quantize_blocks with each scale rounded up to a power of two
    (2^ceil(log2(amax / 448))), returned as its E8M0 byte (exponent + 127)."""
    R, K = x.shape
    RB, KB = -(-R // rows_per_block), -(-K // block)
    pad = torch.zeros(RB * rows_per_block, KB * block, dtype=torch.float32)
    pad[:R, :K] = x
    blocks = pad.view(RB, rows_per_block, KB, block)
    amax = blocks.abs().amax(dim=(1, 3))
    e = torch.where(amax > 0, torch.ceil(torch.log2(amax / 448.0)), torch.zeros_like(amax)).to(torch.int32)
    scale = torch.ldexp(torch.ones_like(amax), e.to(torch.float32))
    q = (blocks / scale[:, None, :, None]).clamp(-448.0, 448.0)
    codes = q.reshape(RB * rows_per_block, KB * block)[:R, :K].contiguous().to(torch.float8_e4m3fn)
    return codes.view(torch.uint8), (e + 127).to(torch.uint8)


def draw_mxfp8_block_scaled(M: int, N: int, K: int, values: str, seed: int):
    """CPU tensors (A codes (M,K) uint8, SA (M,KB) E8M0 bytes, W codes (N,K)
    uint8, SW (NB,KB) E8M0 bytes) for the power-of-two-scale FP8 GEMM, blocks
    of 128: the "normal" recipe of draw_fp8_block_scaled with every scale
    rounded up to a power of two, or small integers with exponents -3..3."""
    g = torch.Generator().manual_seed(int(seed))
    block = FP8_BLOCK
    KB, NB = -(-K // block), -(-N // block)
    if values == "normal":
        a = torch.randn(M, K, generator=g, dtype=torch.float32)
        w = torch.randn(N, K, generator=g, dtype=torch.float32) * (1.0 / math.sqrt(max(K, 1)))
        A, SA = _quantize_blocks_pow2(a, 1, block)
        W, SW = _quantize_blocks_pow2(w, block, block)
        return A, SA, W, SW
    if values == "integer":
        a = torch.randint(-4, 5, (M, K), generator=g, dtype=torch.int32).to(torch.float32)
        w = torch.randint(-4, 5, (N, K), generator=g, dtype=torch.int32).to(torch.float32)
        SA = (torch.randint(-3, 4, (M, KB), generator=g, dtype=torch.int32) + 127).to(torch.uint8)
        SW = (torch.randint(-3, 4, (NB, KB), generator=g, dtype=torch.int32) + 127).to(torch.uint8)
        A = a.to(torch.float8_e4m3fn).view(torch.uint8)
        W = w.to(torch.float8_e4m3fn).view(torch.uint8)
        return A, SA, W, SW
    raise ValueError(f"unknown value recipe {values!r}")


FP8_WORKLOADS: dict[str, Fp8Workload] = {
    "fp8_int_256": Fp8Workload("fp8_int_256", 256, 256, 384, True, "integer", 21),
    "fp8_ragged_1000": Fp8Workload("fp8_ragged_1000", 1000, 1000, 1040, True, "normal", 22),
    "fp8_8192": Fp8Workload("fp8_8192", 8192, 8192, 8192, False, "normal", 23),
}


# ---------------------------------------------------------------------------
# Attention forward operands.  The TileLang-MUSA lesson (section 5) declares
# Q, K, V and O as (batch, heads, seq, dim) float16 buffers; they are drawn
# as the pages draw GEMM operands (torch.randn in float32, rounded to
# float16), Q first, then K, then V, from one generator.


@dataclass(frozen=True)
class AttnWorkload:
    """O = softmax(sm_scale Q K^T [causal]) V per (batch, head)."""
    name: str
    batch: int
    heads: int
    seq: int
    dim: int
    causal: bool
    seed: int

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.dim)

    @property
    def flops(self) -> int:
        # two matmuls of 2 * seq * seq * dim per (batch, head); causal: the
        # half of the score matrix on and below the diagonal
        full = 4 * self.batch * self.heads * self.seq * self.seq * self.dim
        return full // 2 if self.causal else full


def draw_attention(batch: int, heads: int, seq: int, dim: int, seed: int):
    """CPU float16 tensors Q, K, V of shape (batch, heads, seq, dim)."""
    g = torch.Generator().manual_seed(int(seed))
    shape = (batch, heads, seq, dim)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    return q.half(), k.half(), v.half()


def draw_attention_workload(w: AttnWorkload):
    return draw_attention(w.batch, w.heads, w.seq, w.dim, w.seed)


ATTN_WORKLOADS: dict[str, AttnWorkload] = {
    "attn_small_d64": AttnWorkload("attn_small_d64", 1, 2, 200, 64, False, 41),
    "attn_causal_ragged_d128": AttnWorkload("attn_causal_ragged_d128", 2, 3, 300, 128, True, 42),
    "attn_4096_d128": AttnWorkload("attn_4096_d128", 4, 32, 4096, 128, False, 43),
    "attn_4096_d128_causal": AttnWorkload("attn_4096_d128_causal", 4, 32, 4096, 128, True, 44),
    "attn_4096_d64": AttnWorkload("attn_4096_d64", 4, 64, 4096, 64, False, 45),
    "attn_4096_d64_causal": AttnWorkload("attn_4096_d64_causal", 4, 64, 4096, 64, True, 46),
}
