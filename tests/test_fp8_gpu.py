"""GPU parity of the FP8 block-scaled GEMM against the CPU oracle.

Definition (the plainest reading of fp8_block_scaled_linear(x, w_fp8,
scale_w, block=128), TileLang-MUSA lesson, 7yue.com, section 8.2):
C = R(sum_b SA[:,b] SW[n/128,b] (A_b @ W_b^T)), E4M3 A (M,K) and W (N,K),
fp32 scales per row x 128 K (A) and per 128 x 128 block (W), fp16 C.

Bar: bit-exact on integer operands with power-of-two scales (every partial
sum and every scaled sum is exact in fp32, so the only rounding is the final
cast); |gpu - ref| <= 2e-2 + 2e-3 |ref| on quantized N(0,1) operands (the
final fp16 rounding plus fp32 accumulation over the K blocks).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from dense_fp16_gemm_05_gb300.inputs import FP8_WORKLOADS, draw_fp8_block_scaled

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
ATOL, RTOL = 2e-2, 2e-3


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from dense_fp16_gemm_05_gb300 import build as gbuild
    gbuild.build()
    from dense_fp16_gemm_05_gb300 import gemm_f16
    gemm_f16.lib()
    return gemm_f16


def run(g, A, SA, W, SW, relu, C=None):
    out = g.gemm_fp8_block_scaled(A.to(DEV), SA.to(DEV), W.to(DEV), SW.to(DEV), C=C, relu=relu)
    assert g.check() == g.GEMM_OK
    return out.cpu().numpy()


def assert_close(got, ref, what):
    got64, ref64 = got.astype(np.float64), ref.astype(np.float64)
    assert got.shape == ref.shape, what
    assert not np.isnan(got64).any(), what
    err = np.abs(got64 - ref64)
    bad = err > ATOL + RTOL * np.abs(ref64)
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside tolerance, max err {err.max():.4g}"


@pytest.mark.parametrize("relu", [True, False])
def test_integer_workload_bit_exact(g, relu):
    w = FP8_WORKLOADS["fp8_int_256"]
    A, SA, W, SW = draw_fp8_block_scaled(w.M, w.N, w.K, w.values, w.seed)
    ref = oracle.gemm_fp8_block_scaled(A, SA, W, SW, relu=relu)
    got = run(g, A, SA, W, SW, relu)
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))


def test_ragged_normal_full(g):
    w = FP8_WORKLOADS["fp8_ragged_1000"]
    A, SA, W, SW = draw_fp8_block_scaled(w.M, w.N, w.K, w.values, w.seed)
    ref = oracle.gemm_fp8_block_scaled(A, SA, W, SW, relu=True)
    assert_close(run(g, A, SA, W, SW, True), ref, w.name)


def test_8192_sampled_rows(g):
    w = FP8_WORKLOADS["fp8_8192"]
    A, SA, W, SW = draw_fp8_block_scaled(w.M, w.N, w.K, w.values, w.seed)
    got = run(g, A, SA, W, SW, w.relu)
    rng = np.random.default_rng(0)
    rows = sorted({0, 1, 127, 128, 255, 256, 4095, 8191} | set(int(r) for r in rng.integers(0, w.M, 16)))
    ref = oracle.gemm_fp8_block_scaled(A, SA, W, SW, relu=w.relu, rows=rows)
    assert_close(got[rows], ref, w.name)


@pytest.mark.parametrize("M", [1, 127, 129, 257])
@pytest.mark.parametrize("N,K", [(8, 16), (136, 144), (264, 272), (128, 128)])
def test_edge_shapes_integer_bit_exact(g, M, N, K):
    A, SA, W, SW = draw_fp8_block_scaled(M, N, K, "integer", seed=M * 7 + N * 3 + K)
    ref = oracle.gemm_fp8_block_scaled(A, SA, W, SW, relu=True)
    got = run(g, A, SA, W, SW, True)
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16)), (M, N, K)


def test_relu_is_max_of_plain(g):
    A, SA, W, SW = draw_fp8_block_scaled(300, 264, 400, "normal", seed=31)
    on = run(g, A, SA, W, SW, True)
    off = run(g, A, SA, W, SW, False)
    expect = np.where(off > 0, off, np.float16(0))
    assert np.array_equal(on.view(np.uint16), expect.view(np.uint16))


def test_output_guard_bands_untouched(g):
    M, N, K = 200, 264, 272
    A, SA, W, SW = draw_fp8_block_scaled(M, N, K, "normal", seed=33)
    pad = 512
    buf = torch.full((M * N + 2 * pad,), 7.0, dtype=torch.float16, device=DEV)
    C = buf[pad:pad + M * N].view(M, N)
    g.gemm_fp8_block_scaled(A.to(DEV), SA.to(DEV), W.to(DEV), SW.to(DEV), C=C, relu=True)
    assert g.check() == g.GEMM_OK
    assert torch.all(buf[:pad] == 7.0) and torch.all(buf[pad + M * N:] == 7.0)
    assert_close(C.cpu().numpy(), oracle.gemm_fp8_block_scaled(A, SA, W, SW, relu=True), "guarded")


def test_degenerate_and_rejected_arguments(g):
    A, SA, W, SW = draw_fp8_block_scaled(64, 64, 128, "integer", seed=35)
    Ad, SAd, Wd, SWd = A.to(DEV), SA.to(DEV), W.to(DEV), SW.to(DEV)
    # K = 0: C = +0
    C = torch.full((64, 64), 3.0, dtype=torch.float16, device=DEV)
    z8 = torch.empty((64, 0), dtype=torch.uint8, device=DEV)
    zs = torch.empty((64, 0), dtype=torch.float32, device=DEV)
    g.gemm_fp8_block_scaled(z8, zs, z8, torch.empty((1, 0), dtype=torch.float32, device=DEV), C=C)
    assert g.check() == g.GEMM_OK and torch.all(C == 0) and not torch.any(torch.signbit(C))
    # K not a multiple of 16: rejected before any launch
    A2 = torch.zeros((64, 120), dtype=torch.uint8, device=DEV)
    S2 = torch.ones((64, 1), dtype=torch.float32, device=DEV)
    with pytest.raises(g.GemmError) as e:
        g.gemm_fp8_block_scaled(A2, S2, A2, torch.ones((1, 1), dtype=torch.float32, device=DEV))
    assert e.value.status == g.GEMM_ERR_ALIGNMENT
    # C overlapping an input
    big = torch.zeros(64 * 128 + 64 * 64 * 2, dtype=torch.uint8, device=DEV)
    Cov = big[:64 * 64 * 2].view(torch.float16).view(64, 64)
    Aov = big[:64 * 128].view(64, 128)
    with pytest.raises(g.GemmError):
        g.gemm_fp8_block_scaled(Aov, SAd, Wd, SWd, C=Cov)
    assert g.check() == g.GEMM_OK


def test_launch_geometry(g):
    info = g.fp8_launch_info(8192, 8192, 8192)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    assert info["tiles"] == 32 * 32 and info["grid_ctas"] % 2 == 0 and 0 < info["grid_ctas"] <= sms
