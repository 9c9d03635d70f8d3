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
