"""GPU tests of the cluster K split (the configuration for which
gemm_f16_config_cluster_k is 1): the K loop of each 128 x 128 tile runs on the
S CTAs of a cluster (S = 1, 2, 4, 8), and the partial tiles are added in rank
order through distributed shared memory.

* Parity with the oracle within the stated tolerance on ragged shapes, every
  cluster size, ReLU on and off; bit-exact on small-integer operands.
* Bit-identical to the workspace K split of the 128 x 128 configuration with
  the same slices (same per-slice MMA sums, same ascending-rank addition).
* More tiles than resident clusters (one cluster per tile, in waves).
* Guard bands around C, the size rule, and rejected cluster sizes.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from dense_fp16_gemm_05_gb300.inputs import draw

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


@pytest.fixture(scope="module")
def ck(g):
    ids = [c for c in range(1, g.num_configs() + 1) if g.config_cluster_k(c)]
    assert len(ids) == 1
    return ids[0]


def run(g, A, B, relu, config):
    C = g.gemm_f16(A.to(DEV), B.to(DEV), relu=relu, config=config)
    assert g.check() == g.GEMM_OK
    return C.cpu().numpy()


def assert_close(got, ref, what):
    got64, ref64 = got.astype(np.float64), ref.astype(np.float64)
    assert not np.isnan(got64).any(), what
    err = np.abs(got64 - ref64)
    bad = err > ATOL + RTOL * np.abs(ref64)
    assert not bad.any(), f"{what}: {int(bad.sum())} outside tolerance, max err {err.max():.4g}"


@pytest.mark.parametrize("size", [1, 2, 4, 8])
@pytest.mark.parametrize("M,N,K", [(128, 128, 1024), (300, 264, 2056), (1000, 1000, 1000), (64, 8, 4096)])
def test_oracle_parity_every_cluster_size(g, ck, size, M, N, K):
    A, B = draw(M, N, K, "normal_scaled", seed=M + 3 * N + K + size)
    word = ck | (g.ksplit(size) if size > 1 else g.GEMM_F16_NO_KSPLIT)
    for relu in (True, False):
        assert_close(run(g, A, B, relu, word), oracle.gemm_f16(A, B, relu=relu), f"{M}x{N}x{K} S={size} relu={relu}")


@pytest.mark.parametrize("size", [2, 4, 8])
def test_integers_bit_exact(g, ck, size):
    # |partial sums| <= 16 * 2048: exact in fp32; results exact in fp16 where
    # representable, and rounded once like the oracle's
    A, B = draw(256, 200, 2048, "integer", seed=60 + size)
    for relu in (True, False):
        ref = oracle.gemm_f16(A, B, relu=relu)
        got = run(g, A, B, relu, ck | g.ksplit(size))
        assert np.array_equal(got.view(np.uint16), ref.view(np.uint16)), (size, relu)


@pytest.mark.parametrize("size", [2, 4, 8])
def test_same_bits_as_the_workspace_split(g, ck, size):
    # the 128 x 128 workspace configuration with the same slices adds the same
    # per-slice fp32 sums in the same order
    work = [c for c in g.workspace_split_configs() if g.config_name(c).startswith("1sm_128x128")]
    assert work
    A, B = draw(1000, 1032, 3000, "normal", seed=70 + size)
    for relu in (True, False):
        a = run(g, A, B, relu, ck | g.ksplit(size))
        b = run(g, A, B, relu, work[0] | g.ksplit(size))
        assert np.array_equal(a.view(np.uint16), b.view(np.uint16)), (size, relu)


def test_more_tiles_than_resident_clusters(g, ck):
    # 32 x 32 = 1024 tiles, one cluster each: the clusters run in several
    # waves, each reusing SMs that earlier clusters have left
    M = N = 4096
    K = 1024
    A, B = draw(M, N, K, "normal_scaled", seed=81)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    info = g.launch_info(M, N, K, ck | g.ksplit(2))
    assert info["cluster_size"] == 2 and info["grid_ctas"] == 2 * info["tiles"] > 4 * sms
    got = run(g, A, B, True, ck | g.ksplit(2))
    rows = [0, 1, 127, 128, 129, 2047, 2048, 4000, 4095]
    assert_close(got[rows], oracle.gemm_f16(A, B, relu=True, rows=rows), "4096^2 x 1024, S=2")
    work = [c for c in g.workspace_split_configs() if g.config_name(c).startswith("1sm_128x128")][0]
    again = run(g, A, B, True, work | g.ksplit(2))
    assert np.array_equal(got.view(np.uint16), again.view(np.uint16))


def test_guard_bands_untouched(g, ck):
    M, N, K = 200, 136, 1504
    A, B = draw(M, N, K, "normal_scaled", seed=90)
    ref = oracle.gemm_f16(A, B, relu=True)
    pad = 512
    for size in (2, 4, 8):
        buf = torch.full((M * N + 2 * pad,), 7.0, dtype=torch.float16, device=DEV)
        # C starts 16-byte aligned inside the buffer
        C = buf[pad:pad + M * N].view(M, N)
        g.gemm_f16(A.to(DEV), B.to(DEV), C, relu=True, config=ck | g.ksplit(size))
        assert g.check() == g.GEMM_OK
        assert torch.all(buf[:pad] == 7.0) and torch.all(buf[pad + M * N:] == 7.0)
        assert_close(C.cpu().numpy(), ref, f"guard S={size}")


def test_size_rule_and_launch_geometry(g, ck):
    # 512^3: 16 tiles, 8 K blocks -> clusters of 4 (8 would leave one block per CTA)
    info = g.launch_info(512, 512, 512, ck)
    assert info["tiles"] == 16 and info["cluster_size"] == 4 and info["grid_ctas"] == 64
    # 1024 x 1024 x 16384: 64 tiles -> clusters of 2 fill 128 SMs
    info = g.launch_info(1024, 1024, 16384, ck)
    assert info["cluster_size"] == 2 and info["grid_ctas"] == 128
    # many tiles: no split (one CTA per tile)
    info = g.launch_info(8192, 8192, 8192, ck)
    assert info["cluster_size"] == 1 and info["grid_ctas"] == info["tiles"] == 64 * 64
    # a short K halves the requested size until every CTA has a block
    assert g.launch_info(256, 256, 192, ck | g.ksplit(8))["cluster_size"] == 2
    # a resolved automatic choice names its cluster size in the word
    c = g.auto_config(512, 512, 512)
    if g.config_cluster_k(c):
        n = (c & g.GEMM_F16_KSPLIT_MASK) >> g.GEMM_F16_KSPLIT_SHIFT
        assert g.launch_info(512, 512, 512, c)["cluster_size"] == max(n, 1)


def test_rejected_sizes_launch_nothing(g, ck):
    A, B = (x.to(DEV) for x in draw(128, 128, 1024, "normal", seed=1))
    C = torch.full((128, 128), 3.0, dtype=torch.float16, device=DEV)
    for word in (ck | g.ksplit(3), ck | g.ksplit(16), ck | g.GEMM_F16_KSPLIT_TAIL):
        with pytest.raises(g.GemmError) as e:
            g.gemm_f16(A, B, C, config=word)
        assert e.value.status == g.GEMM_ERR_INVALID_ARG
    with pytest.raises(g.GemmError):
        g.gemm_f16_t(A, B.t().contiguous(), C, transb=True, config=ck)   # NN layout only
    torch.cuda.synchronize()
    assert torch.all(C == 3.0)
    assert g.check() == g.GEMM_OK
