"""GPU parity of the FP8 GEMM with power-of-two block scales against the CPU oracle.

Definition: C = R(sum_b 2^(SA[i,b]-127) 2^(SW[n/128,b]-127) (A_b @ W_b^T)),
the FP8 block-scaled linear layer of the TileLang-MUSA lesson (7yue.com,
section 8.2, blocks of 128) with every scale a power of two given as its
E8M0 byte; E4M3 A (M,K) and W (N,K), fp16 C.  The kernel applies the scales
inside the tensor core (block-scaled MMA) and accumulates all K blocks in
one fp32 accumulator.

Bar: bit-exact on integer operands (every product and partial sum is exact
in fp32, the scales are powers of two, so the only rounding is the final
cast); |gpu - ref| <= 2e-2 + 2e-3 |ref| on quantized N(0,1) operands.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from dense_fp16_gemm_05_gb300.inputs import draw_mxfp8_block_scaled

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
    out = g.gemm_mxfp8_block_scaled(A.to(DEV), SA.to(DEV), W.to(DEV), SW.to(DEV), C=C, relu=relu)
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
def test_integer_operands_bit_exact(g, relu):
    A, SA, W, SW = draw_mxfp8_block_scaled(256, 512, 384, "integer", 31)
    ref = oracle.gemm_mxfp8_block_scaled(A, SA, W, SW, relu=relu)
    got = run(g, A, SA, W, SW, relu)
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))


@pytest.mark.parametrize("M", [1, 127, 129, 257])
@pytest.mark.parametrize("N,K", [(8, 16), (136, 144), (264, 272), (128, 128), (520, 1040)])
def test_edge_shapes_bit_exact(g, M, N, K):
    A, SA, W, SW = draw_mxfp8_block_scaled(M, N, K, "integer", M + N + K)
    ref = oracle.gemm_mxfp8_block_scaled(A, SA, W, SW, relu=False)
    got = run(g, A, SA, W, SW, False)
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16)), (M, N, K)


def test_ragged_normal_full(g):
    A, SA, W, SW = draw_mxfp8_block_scaled(1000, 1000, 1040, "normal", 32)
    ref = oracle.gemm_mxfp8_block_scaled(A, SA, W, SW, relu=True)
    assert_close(run(g, A, SA, W, SW, True), ref, "1000x1000x1040")


def test_8192_sampled_rows(g):
    A, SA, W, SW = draw_mxfp8_block_scaled(8192, 8192, 8192, "normal", 33)
    got = run(g, A, SA, W, SW, False)
    rng = np.random.default_rng(1)
    rows = sorted({0, 1, 127, 128, 255, 256, 4095, 8191} | set(int(r) for r in rng.integers(0, 8192, 12)))
    ref = oracle.gemm_mxfp8_block_scaled(A, SA, W, SW, relu=False, rows=rows)
    assert_close(got[rows], ref, "8192^3")


def test_relu_is_max_of_plain(g):
    A, SA, W, SW = draw_mxfp8_block_scaled(384, 768, 2048, "normal", 34)
    plain = run(g, A, SA, W, SW, False)
    relu = run(g, A, SA, W, SW, True)
    expect = np.where(plain.astype(np.float64) > 0, plain, np.float16(0.0)).astype(np.float16)
    assert np.array_equal(relu.view(np.uint16), expect.view(np.uint16))


def test_matches_the_fp32_scale_kernel(g):
    # the same problem through gemm_fp8_block_scaled with the decoded scales
    A, SA, W, SW = draw_mxfp8_block_scaled(512, 640, 1536, "normal", 35)
    mx = run(g, A, SA, W, SW, True)
    sa = torch.from_numpy(oracle.e8m0_to_f32(SA.numpy()))
    sw = torch.from_numpy(oracle.e8m0_to_f32(SW.numpy()))
    f32 = g.gemm_fp8_block_scaled(A.to(DEV), sa.to(DEV), W.to(DEV), sw.to(DEV), relu=True).cpu().numpy()
    assert g.check() == g.GEMM_OK
    assert_close(mx, f32, "power-of-two scales vs fp32 scales")


def test_guard_bands_and_empty(g):
    M, N, K = 200, 136, 400
    A, SA, W, SW = draw_mxfp8_block_scaled(M, N, K, "integer", 36)
    pad = 512
    buf = torch.full((M * N + 2 * pad,), 7.0, dtype=torch.float16, device=DEV)
    C = buf[pad:pad + M * N].view(M, N)
    g.gemm_mxfp8_block_scaled(A.to(DEV), SA.to(DEV), W.to(DEV), SW.to(DEV), C=C, relu=True)
    assert g.check() == g.GEMM_OK
    assert torch.all(buf[:pad] == 7.0) and torch.all(buf[pad + M * N:] == 7.0)
    ref = oracle.gemm_mxfp8_block_scaled(A, SA, W, SW, relu=True)
    assert np.array_equal(C.cpu().numpy().view(np.uint16), ref.view(np.uint16))
    # K = 0: the empty sum, +0 everywhere
    z = torch.full((4, 8), 5.0, dtype=torch.float16, device=DEV)
    e8 = torch.empty((4, 0), dtype=torch.uint8, device=DEV)
    g.gemm_mxfp8_block_scaled(e8, torch.empty((4, 0), dtype=torch.uint8, device=DEV),
                              torch.empty((8, 0), dtype=torch.uint8, device=DEV),
                              torch.empty((1, 0), dtype=torch.uint8, device=DEV), C=z, relu=False)
    assert g.check() == g.GEMM_OK
    assert torch.all(z.view(torch.int16) == 0)


def test_rejected_arguments(g):
    L = g.lib()
    assert L.gemm_mxfp8_block_scaled(None, None, None, None, None, -1, 8, 16, 1, None) == g.GEMM_ERR_INVALID_ARG
    assert L.gemm_mxfp8_block_scaled(None, None, None, None, None, 8, 8, 16, 2, None) == g.GEMM_ERR_INVALID_ARG
    A = torch.zeros((8, 24), dtype=torch.uint8, device=DEV)
    W = torch.zeros((8, 24), dtype=torch.uint8, device=DEV)
    S = torch.zeros((8, 1), dtype=torch.uint8, device=DEV)
    C = torch.zeros((8, 8), dtype=torch.float16, device=DEV)
    # K not a multiple of 16
    assert L.gemm_mxfp8_block_scaled(A.data_ptr(), S.data_ptr(), W.data_ptr(), S.data_ptr(), C.data_ptr(),
                                     8, 8, 24, 1, None) == g.GEMM_ERR_ALIGNMENT
    assert g.check() == g.GEMM_OK
