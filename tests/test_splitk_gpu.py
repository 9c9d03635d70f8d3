"""GPU parity of the K-split GEMM path against the CPU oracle.

Same definition and tolerance as tests/test_gemm_gpu.py (C = R(A @ B) of the
tile GEMM in "Writing High-Performance Kernels in TileLang, from GEMM to MLA",
"Let's write a GEMM"; |gpu - ref| <= 2e-2 + 2e-3 |ref|): a K split changes
only the order in which the fp32 partial sums are added.  Integer operands
small enough that every partial sum is exact give bit-identical results with
and without a split; ReLU stays bitwise max(plain, +0).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from dense_fp16_gemm_05_gb300.inputs import draw

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-2, 2e-3
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


def run(g, A, B, relu, config):
    C = g.gemm_f16(A.to(DEV), B.to(DEV), relu=relu, config=config)
    assert g.check() == g.GEMM_OK
    return C.cpu().numpy()


def assert_close(got, ref, what=""):
    got64, ref64 = got.astype(np.float64), ref.astype(np.float64)
    assert got.shape == ref.shape, what
    assert not np.isnan(got64).any(), f"{what}: NaN"
    err = np.abs(got64 - ref64)
    bad = err > ATOL + RTOL * np.abs(ref64)
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside tolerance, max err {err.max():.4g}"


SHAPES = [(128, 128, 4096), (256, 136, 1000), (300, 264, 2056), (64, 520, 8192)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("splits", [2, 3, 5, 16])
def test_explicit_splits_every_config(g, M, N, K, splits):
    A, B = draw(M, N, K, "normal_scaled", seed=M + N + K + splits)
    for relu in (True, False):
        ref = oracle.gemm_f16(A, B, relu=relu)
        for cfg in g.workspace_split_configs():
            got = run(g, A, B, relu, cfg | g.ksplit(splits))
            assert_close(got, ref, f"{M}x{N}x{K} cfg {cfg} splits {splits} relu {relu}")


@pytest.mark.parametrize("splits", [2, 7, 16])
def test_integers_bit_exact_with_and_without_split(g, splits):
    # |partial sums| <= 16 * K, exact in fp32 and fp16 for K = 2048
    A, B = draw(192, 264, 2048, "integer", seed=5 + splits)
    for relu in (True, False):
        ref = oracle.gemm_f16(A, B, relu=relu)
        whole = run(g, A, B, relu, 3 | g.GEMM_F16_NO_KSPLIT)
        cut = run(g, A, B, relu, 3 | g.ksplit(splits))
        assert np.array_equal(whole.view(np.uint16), cut.view(np.uint16)), (splits, relu)
        # bit for bit with and without ReLU: an exact zero sum is +0
        assert np.array_equal(cut.view(np.uint16), ref.view(np.uint16))


def test_relu_is_max_of_plain_with_split(g):
    A, B = draw(256, 256, 4096, "normal", seed=91)
    for cfg in (2, 3):
        plain = run(g, A, B, False, cfg | g.ksplit(6))
        relu = run(g, A, B, True, cfg | g.ksplit(6))
        expect = np.where(plain.astype(np.float64) > 0, plain, np.float16(0.0)).astype(np.float16)
        assert np.array_equal(relu.view(np.uint16), expect.view(np.uint16)), cfg


@pytest.mark.parametrize("transa,transb", [(False, True), (True, False), (True, True)])
def test_transposed_layouts_with_split(g, transa, transb):
    M, N, K = 192, 200, 3000
    A, B = draw(M, N, K, "normal_scaled", seed=17 + 2 * transa + transb)
    As = A.t().contiguous() if transa else A
    Bs = B.t().contiguous() if transb else B
    ref = oracle.gemm_f16(A, B, relu=True)
    for cfg in g.workspace_split_configs():
        if g.config_layouts(cfg) != 0xF:
            continue
        C = g.gemm_f16_t(As.to(DEV), Bs.to(DEV), transa=transa, transb=transb, relu=True, config=cfg | g.ksplit(4))
        assert g.check() == g.GEMM_OK
        assert_close(C.cpu().numpy(), ref, f"cfg {cfg} transa {transa} transb {transb}")


def test_more_splits_than_k_blocks(g):
    # K = 64 is one block: no split takes place, the result is the one-pass one
    A, B = draw(128, 256, 64, "normal", seed=3)
    whole = run(g, A, B, True, 2 | g.GEMM_F16_NO_KSPLIT)
    cut = run(g, A, B, True, 2 | g.ksplit(16))
    assert np.array_equal(whole.view(np.uint16), cut.view(np.uint16))
    # K = 200 has 4 blocks (the last partial): 16 requested -> 4 slices
    A, B = draw(128, 256, 200, "normal_scaled", seed=4)
    assert_close(run(g, A, B, True, 2 | g.ksplit(16)), oracle.gemm_f16(A, B, relu=True), "K=200")


def test_rule_chosen_split_on_few_tiles(g):
    # configuration 2 (128 x 128 tiles) has 64 tiles at 1024 x 1024 for 152
    # slots: the rule cuts K = 16384 (256 blocks) into 152 // 64 = 2 slices
    M, N, K = 1024, 1024, 16384
    cfg = 2 | g.GEMM_F16_KSPLIT_AUTO
    assert g.launch_info(M, N, K, cfg)["grid_ctas"] == 128
    assert g.launch_info(8192, 8192, 8192, cfg)["grid_ctas"] == g.launch_info(8192, 8192, 8192, 2)["grid_ctas"]
    A, B = draw(M, N, K, "normal_scaled", seed=44)
    got = run(g, A, B, True, cfg)
    rows = [0, 1, 127, 128, 511, 512, 1000, 1023]
    ref = oracle.gemm_f16(A, B, relu=True, rows=rows)
    assert_close(got[rows], ref, "rule split 1024x1024x16384")
    again = run(g, A, B, True, 2 | g.ksplit(2))
    assert np.array_equal(got.view(np.uint16), again.view(np.uint16))


def test_automatic_choice_reproduces_itself(g):
    # whatever the automatic choice is (never a workspace K split: gemm_f16
    # allocates nothing), passing it back explicitly computes the same bits
    for (M, N, K) in [(1024, 1024, 16384), (256, 4096, 8192), (2048, 2048, 2048)]:
        c = g.auto_config(M, N, K)
        assert c & (g.GEMM_F16_KSPLIT_AUTO | g.GEMM_F16_KSPLIT_TAIL) == 0
        if not g.config_cluster_k(c):
            assert c & g.GEMM_F16_KSPLIT_MASK == 0
        A, B = draw(M, N, K, "normal_scaled", seed=M + K)
        auto = run(g, A, B, True, 0)
        fixed = run(g, A, B, True, c)
        assert np.array_equal(auto.view(np.uint16), fixed.view(np.uint16)), hex(c)
        rows = [0, M // 2, M - 1]
        assert_close(auto[rows], oracle.gemm_f16(A, B, relu=True, rows=rows), f"auto {M}x{N}x{K}")


def test_guard_bands_untouched(g):
    M, N, K = 160, 136, 3000
    A, B = draw(M, N, K, "normal_scaled", seed=8)
    pad = 4096
    buf = torch.full((M * N + 2 * pad,), 7.0, dtype=torch.float16, device=DEV)
    C = buf[pad:pad + M * N].view(M, N)
    g.gemm_f16(A.to(DEV), B.to(DEV), C=C, relu=True, config=2 | g.ksplit(5))
    assert g.check() == g.GEMM_OK
    assert torch.all(buf[:pad] == 7.0) and torch.all(buf[pad + M * N:] == 7.0)
    assert_close(C.cpu().numpy(), oracle.gemm_f16(A, B, relu=True), "guarded")


def test_split_inside_a_cuda_graph(g):
    # the workspace comes from the stream-ordered allocator, which a stream
    # capture records as allocation nodes; the replayed graph recomputes C
    M, N, K = 256, 256, 8192
    A, B = draw(M, N, K, "normal_scaled", seed=12)
    Ad, Bd = A.to(DEV), B.to(DEV)
    C = torch.empty((M, N), dtype=torch.float16, device=DEV)
    cfg = 2 | g.ksplit(8)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g.gemm_f16(Ad, Bd, C=C, relu=True, config=cfg)      # first call outside the capture
    torch.cuda.synchronize()
    assert g.check() == g.GEMM_OK
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        g.gemm_f16(Ad, Bd, C=C, relu=True, config=cfg)
    C.fill_(0)
    graph.replay()
    torch.cuda.synchronize()
    assert g.check() == g.GEMM_OK
    assert_close(C.cpu().numpy(), oracle.gemm_f16(A, B, relu=True), "graph replay")


def test_launch_info_counts_slices(g):
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    plain = g.launch_info(256, 256, 16384, 2 | g.GEMM_F16_NO_KSPLIT | g.GEMM_F16_NO_SPLIT)
    cut = g.launch_info(256, 256, 16384, 2 | g.ksplit(8))
    assert plain["tiles"] == cut["tiles"] == 4
    assert plain["grid_ctas"] == 4 and cut["grid_ctas"] == 32 <= sms


def test_tail_split_integers_bit_exact(g):
    # configuration 2 (128 x 128 tiles) at 1920 x 1920: 225 tiles, 152 slots,
    # so the last 73 tiles run as 2 K slices each; exact integer sums give the
    # same bits as whole tiles and as the oracle
    A, B = draw(1920, 1920, 2048, "integer", seed=61)
    whole = run(g, A, B, True, 2 | g.GEMM_F16_NO_SPLIT | g.GEMM_F16_NO_KSPLIT)
    tail = run(g, A, B, True, 2 | g.GEMM_F16_KSPLIT_TAIL)
    assert np.array_equal(whole.view(np.uint16), tail.view(np.uint16))
    rows = [0, 640, 1279, 1280, 1700, 1919]
    assert np.array_equal(tail[rows].view(np.uint16), oracle.gemm_f16(A, B, relu=True, rows=rows).view(np.uint16))


@pytest.mark.parametrize("cfg", [1, 2, 3, 5])
def test_tail_split_normal_values(g, cfg):
    M, N, K = 2300, 1800, 3000
    A, B = draw(M, N, K, "normal_scaled", seed=62 + cfg)
    got = run(g, A, B, True, cfg | g.GEMM_F16_KSPLIT_TAIL)
    rows = sorted(set([0, 255, 256, 1023, 1024, 2047, 2048, 2299] + list(range(2200, 2300, 7))))
    assert_close(got[rows], oracle.gemm_f16(A, B, relu=True, rows=rows), f"tail split cfg {cfg}")


def test_tail_split_headline_shape(g):
    A, B = draw(8192, 8192, 8192, "normal_scaled", seed=5)
    got = run(g, A, B, True, 5 | g.GEMM_F16_KSPLIT_TAIL)
    rows = [0, 4095, 7680, 7935, 7936, 8191]
    assert_close(got[rows], oracle.gemm_f16(A, B, relu=True, rows=rows), "tail split 8192^3")
