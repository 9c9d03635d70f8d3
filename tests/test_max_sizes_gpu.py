"""GPU tests at sizes past 2^31 elements (the edge of 32-bit index arithmetic).

Each kernel writes an output with more than 2^31 elements (4-17 GB on the
device); sampled rows at the start, the middle and the very end are compared
with the oracle, which gets the same inputs drawn on the CPU.  A 32-bit
overflow anywhere in the address arithmetic (row * N, flat element index,
head offset) would misplace or drop the late rows.

Tolerances as in the per-kernel tests: bit-exact on integer GEMM inputs and
for the ReLU gradient; |gpu - ref| <= 2e-2 + 2e-3 |ref| for FP8 and
6e-3 + 2e-3 |ref| for attention.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from dense_fp16_gemm_05_gb300.inputs import draw, draw_attention, draw_fp8_block_scaled

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from dense_fp16_gemm_05_gb300 import build as gbuild
    gbuild.build()
    from dense_fp16_gemm_05_gb300 import gemm_f16
    gemm_f16.lib()
    return gemm_f16


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def edge_rows(M, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 255, 256, M // 2 - 1, M // 2, M - 257, M - 256, M - 2, M - 1]
    return sorted(set(fixed) | set(int(r) for r in rng.integers(0, M, 6)))


def test_gemm_output_past_2_31_elements(g):
    M, N, K = 65536, 36864, 64                # C: 2.42e9 elements, 4.8 GB
    assert M * N > 2**31
    A, B = draw(M, N, K, "integer", seed=91)  # |partial sums| <= 16 * 64: exact
    Ad, Bd = A.to(DEV), B.to(DEV)
    C = torch.empty((M, N), dtype=torch.float16, device=DEV)
    rows = edge_rows(M, 92)
    ref = oracle.gemm_f16(A, B, relu=True, rows=rows)
    for cfg in [0] + list(range(1, g.num_configs() + 1)):
        C.fill_(float("nan"))
        g.gemm_f16(Ad, Bd, C=C, relu=True, config=cfg)
        assert g.check() == g.GEMM_OK
        got = C[torch.tensor(rows, device=DEV)].cpu().numpy()
        assert np.array_equal(got.view(np.uint16), ref.view(np.uint16)), f"config {cfg}"


def test_relu_backward_past_2_31_elements(g):
    n = 2**31 + 4096 + 5                      # a scalar tail past the vector part too
    cpu = torch.Generator().manual_seed(93)
    block = 1 << 20
    # one CPU-drawn block repeated over the whole length, then CPU-drawn
    # values of their own at the sampled positions
    base_c = torch.randn(block, generator=cpu).half()
    base_g = torch.randn(block, generator=cpu).half()
    C = base_c.to(DEV).repeat(n // block + 1)[:n].contiguous()
    dC = base_g.to(DEV).repeat(n // block + 1)[:n].contiguous()
    idx = [0, 1, 2**31 - 8, 2**31 - 1, 2**31, 2**31 + 1, n - 6, n - 5, n - 2, n - 1]
    c_s = torch.randn(len(idx), generator=cpu).half()
    g_s = torch.randn(len(idx), generator=cpu).half()
    c_s[:3] = torch.tensor([0.0, -0.0, float("inf")]).half()   # the zero / sign / inf cases
    idx_d = torch.tensor(idx, device=DEV)
    C[idx_d] = c_s.to(DEV)
    dC[idx_d] = g_s.to(DEV)
    dZ = g.relu_backward(dC, C)
    assert g.check() == g.GEMM_OK
    ref = oracle.relu_backward(g_s.numpy(), c_s.numpy())
    got = dZ[idx_d].cpu().numpy()
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))


def test_fp8_output_past_2_31_elements(g):
    M, N, K = 65536, 36864, 128
    A, SA, W, SW = draw_fp8_block_scaled(M, N, K, "normal", seed=94)
    out = g.gemm_fp8_block_scaled(A.to(DEV), SA.to(DEV), W.to(DEV), SW.to(DEV), relu=True)
    assert g.check() == g.GEMM_OK
    rows = edge_rows(M, 95)
    got = out[torch.tensor(rows, device=DEV)].cpu().numpy().astype(np.float64)
    ref = oracle.gemm_fp8_block_scaled(A, SA, W, SW, relu=True, rows=rows).astype(np.float64)
    bad = np.abs(got - ref) > 2e-2 + 2e-3 * np.abs(ref)
    assert not bad.any(), f"{int(bad.sum())} outside tolerance"


def test_attention_head_offsets_past_2_31_elements(g):
    # batch 128 x heads 136 x seq 1024 x dim 128 = 2.28e9 elements per tensor.
    # Every head holds one shared CPU-drawn block except the sampled heads,
    # which hold their own draws: a read from the wrong head changes their rows.
    Bn, H, S, D = 128, 136, 1024, 128
    assert Bn * H * S * D > 2**31
    q0, k0, v0 = draw_attention(1, 1, S, D, seed=96)
    Q = q0.to(DEV).expand(Bn, H, S, D).contiguous()
    K = k0.to(DEV).expand(Bn, H, S, D).contiguous()
    V = v0.to(DEV).expand(Bn, H, S, D).contiguous()
    sampled = [(0, 0), (0, 135), (64, 63), (127, 0), (127, 135)]
    own = {}
    for i, (b, h) in enumerate(sampled):
        q, k, v = draw_attention(1, 1, S, D, seed=97 + i)
        own[(b, h)] = (q, k, v)
        Q[b, h], K[b, h], V[b, h] = q[0, 0].to(DEV), k[0, 0].to(DEV), v[0, 0].to(DEV)
    for causal in (False, True):
        O = g.attention_fwd(Q, K, V, causal=causal)
        assert g.check() == g.GEMM_OK
        rows = [0, 1, 127, 128, 511, 1000, 1023]
        for (b, h), (q, k, v) in own.items():
            ref = oracle.attention_fwd(q, k, v, sm_scale=D ** -0.5, causal=causal, rows=rows).astype(np.float64)
            got = O[b, h, rows].cpu().numpy().astype(np.float64)
            bad = np.abs(got - ref) > 6e-3 + 2e-3 * np.abs(ref)
            assert not bad.any(), f"head ({b}, {h}) causal {causal}: {int(bad.sum())} outside tolerance"
        del O
