"""GPU parity tests: the sm_103a kernels (through the C ABI) against the CPU oracle.

Bar (stated by the benchmark description for seeded N(0,1) inputs):
    |C_gpu - C_ref| <= 2e-2 + 2e-3 * |C_ref|   elementwise,
and bit-exact equality on integer-valued inputs, where every product and
partial sum is exact in fp32 and the only rounding is the final (exact) cast.

Sizes the oracle finishes in seconds are compared in full; the large
configurations are compared on sampled full rows (tile edges plus seeded
random rows), in the same launch configuration the bench times.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from dense_fp16_gemm_05_gb300.inputs import WORKLOADS, draw, draw_workload

pytestmark = pytest.mark.gpu

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


DEV = torch.device("cuda:0")


def run(g, A, B, relu, config=0):
    C = g.gemm_f16(A.to(DEV), B.to(DEV), relu=relu, config=config)
    assert g.check() == g.GEMM_OK
    return C.cpu().numpy()


def assert_close(got, ref, what=""):
    got64 = got.astype(np.float64)
    ref64 = ref.astype(np.float64)
    assert got.shape == ref.shape
    assert not np.isnan(got64).any(), f"{what}: NaN in GPU output"
    err = np.abs(got64 - ref64)
    tol = ATOL + RTOL * np.abs(ref64)
    bad = err > tol
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first at {tuple(i)}: "
                             f"gpu {got64[tuple(i)]} ref {ref64[tuple(i)]}; max err {err.max():.4g}")


def sample_rows(M, n_random=24, seed=0):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 31, 32, 127, 128, 129, 255, 256, M // 2, M - 129, M - 128, M - 2, M - 1]
    rows = set(r for r in fixed if 0 <= r < M)
    rows.update(int(r) for r in rng.integers(0, M, n_random))
    return sorted(rows)


def configs(g):
    return list(range(1, g.num_configs() + 1))


# ---------------------------------------------------------------- benchmark configurations

@pytest.mark.parametrize("relu", [True, False])
def test_int64_bit_exact(g, relu):
    w = WORKLOADS["int_64"]
    A, B = draw_workload(w)
    ref = oracle.gemm_f16(A, B, relu=relu)
    for cfg in configs(g):
        got = run(g, A, B, relu, cfg)
        # bit for bit, zero signs included: every exact zero sum is +0 (the
        # accumulator starts at +0), with or without ReLU
        assert np.array_equal(got.view(np.uint16), ref.view(np.uint16)), cfg


@pytest.mark.parametrize("ksplit", [0, 4])
def test_zero_sums_are_plus_zero_without_relu(g, ksplit):
    # Sums that are exactly zero: all terms -0 (a -0 row times a positive
    # column), exact cancellation of +-1 terms, and zeros mixed in.  The
    # oracle's sum starts at +0 (the cleared accumulator of the pages' tile
    # GEMM), so each of these is +0 (0x0000); a -0 would fail the bit test.
    M, N, K = 300, 264, 448
    rng = np.random.default_rng(81)
    a = rng.integers(-4, 5, (M, K)).astype(np.float16)
    b = rng.integers(-4, 5, (K, N)).astype(np.float16)
    a[0::3, :] = np.float16(-0.0)                          # every product -0 against b >= 0
    b[:, 0::2] = np.abs(b[:, 0::2])
    a[1::3, :] = np.where(np.arange(K) % 2 == 0, 1.0, -1.0).astype(np.float16)
    b[:, 1::4] = 1.0                                       # alternating +-1 terms cancel exactly
    A, B = torch.from_numpy(a), torch.from_numpy(b)
    ref = oracle.gemm_f16(A, B, relu=False)
    assert np.count_nonzero(ref.view(np.uint16) == 0) > M * N // 6
    assert not np.any(ref.view(np.uint16) == 0x8000)
    for cfg in configs(g):
        got = run(g, A, B, False, cfg | (g.ksplit(ksplit) if ksplit else 0))
        assert np.array_equal(got.view(np.uint16), ref.view(np.uint16)), (cfg, ksplit)


def test_relu_1024_full(g):
    w = WORKLOADS["relu_1024"]
    A, B = draw_workload(w)
    assert_close(run(g, A, B, True), oracle.gemm_f16(A, B, relu=True), w.name)


def test_ragged_1000_full_all_configs(g):
    w = WORKLOADS["relu_ragged_1000"]
    A, B = draw_workload(w)
    ref = oracle.gemm_f16(A, B, relu=True)
    for cfg in configs(g):
        assert_close(run(g, A, B, True, cfg), ref, f"{w.name} cfg {cfg}")


def test_plain_4096_sampled(g):
    w = WORKLOADS["plain_4096"]
    A, B = draw_workload(w)
    got = run(g, A, B, False)
    rows = sample_rows(w.M, seed=4)
    assert_close(got[rows], oracle.gemm_f16(A, B, relu=False, rows=rows), w.name)
    assert np.isfinite(got.astype(np.float32)).all()
    assert (got.astype(np.float32) < 0).any()   # no ReLU applied


def test_relu_8192_sampled(g):
    w = WORKLOADS["relu_8192"]
    A, B = draw_workload(w)
    got = run(g, A, B, True)
    rows = sample_rows(w.M, seed=5)
    assert_close(got[rows], oracle.gemm_f16(A, B, relu=True, rows=rows), w.name)
    assert (got.view(np.uint16) & 0x8000 == 0).all()   # ReLU output has no sign bit set


@pytest.mark.parametrize("n", [512, 1024, 2048, 4096, 16384])
def test_sweep(g, n):
    w = WORKLOADS[f"sweep_{n}"]
    A, B = draw_workload(w)
    got = run(g, A, B, True)
    if n <= 2048:
        assert_close(got, oracle.gemm_f16(A, B, relu=True), w.name)
    else:
        rows = sample_rows(n, n_random=12 if n > 8192 else 24, seed=n)
        assert_close(got[rows], oracle.gemm_f16(A, B, relu=True, rows=rows), w.name)


# ---------------------------------------------------------------- edges and invariants

EDGE_MN = [(1, 8), (7, 120), (127, 128), (128, 136), (129, 248), (255, 256), (257, 264), (64, 520)]
EDGE_K = [8, 56, 64, 72, 200]


@pytest.mark.parametrize("M,N", EDGE_MN)
@pytest.mark.parametrize("K", EDGE_K)
def test_edge_shapes(g, M, N, K):
    A, B = draw(M, N, K, "normal", seed=M * 1000 + N + K)
    ref = oracle.gemm_f16(A, B, relu=True)
    for cfg in configs(g):
        assert_close(run(g, A, B, True, cfg), ref, f"{M}x{N}x{K} cfg {cfg}")


def test_relu_is_max_of_plain_bitwise(g):
    A, B = draw(1000, 1000, 1000, "normal", seed=21)
    for cfg in configs(g):
        plain = run(g, A, B, False, cfg)
        relu = run(g, A, B, True, cfg)
        want = np.where(plain.astype(np.float32) > 0, plain, np.float16(0)).astype(np.float16)
        assert np.array_equal(relu.view(np.uint16), want.view(np.uint16)), cfg


def test_guard_bands_untouched(g):
    M, N, K = 300, 264, 136
    A, B = draw(M, N, K, "normal", seed=22)
    pad = 512  # elements = 1 KiB each side
    buf = torch.full((pad + M * N + pad,), -7.0, dtype=torch.float16, device=DEV)
    C = buf[pad:pad + M * N].view(M, N)
    for cfg in configs(g):
        g.gemm_f16(A.to(DEV), B.to(DEV), C, relu=True, config=cfg)
        assert g.check() == g.GEMM_OK
        host = buf.cpu()
        assert torch.all(host[:pad] == -7.0) and torch.all(host[pad + M * N:] == -7.0)
        assert_close(C.cpu().numpy(), oracle.gemm_f16(A, B, relu=True), f"cfg {cfg}")


def test_k_zero_fills_plus_zero(g):
    A = torch.zeros((5, 0), dtype=torch.float16, device=DEV)
    B = torch.zeros((0, 8), dtype=torch.float16, device=DEV)
    C = torch.full((5, 8), 3.0, dtype=torch.float16, device=DEV)
    g.gemm_f16(A, B, C, relu=False)
    assert g.check() == g.GEMM_OK
    assert np.all(C.cpu().numpy().view(np.uint16) == 0)


def test_empty_m_is_no_op(g):
    A = torch.zeros((0, 8), dtype=torch.float16, device=DEV)
    B = torch.zeros((8, 8), dtype=torch.float16, device=DEV)
    C = g.gemm_f16(A, B, relu=True)
    assert C.shape == (0, 8)


def test_runs_on_the_given_stream(g):
    A, B = draw(256, 256, 256, "normal", seed=23)
    s = torch.cuda.Stream(device=DEV)
    with torch.cuda.stream(s):
        Ad, Bd = A.to(DEV), B.to(DEV)
        C = g.gemm_f16(Ad, Bd, relu=True, stream=s)
    s.synchronize()
    assert_close(C.cpu().numpy(), oracle.gemm_f16(A, B, relu=True), "side stream")


def test_from_host_matches_oracle(g):
    M, N, K = 384, 512, 320
    A, B = draw(M, N, K, "normal", seed=24)
    Ah, Bh = A.pin_memory(), B.pin_memory()
    Ch = torch.empty((M, N), dtype=torch.float16).pin_memory()
    Ad = torch.empty_like(A, device=DEV)
    Bd = torch.empty_like(B, device=DEV)
    Cd = torch.empty((M, N), dtype=torch.float16, device=DEV)
    g.gemm_f16_from_host(Ah, Bh, Ch, Ad, Bd, Cd, relu=True)
    torch.cuda.synchronize()
    assert g.check() == g.GEMM_OK
    assert_close(Ch.numpy(), oracle.gemm_f16(A, B, relu=True), "from_host")


@pytest.mark.parametrize("M", [3000, 4096, 9000])
def test_from_host_row_panels(g, M):
    # 2, 4 and 8 row panels (the last one ragged for 3000 and 9000); the side
    # stream alone covers uploads, GEMMs and downloads
    N, K = 264, 520
    A, B = draw(M, N, K, "normal_scaled", seed=M)
    Ah, Bh = A.pin_memory(), B.pin_memory()
    Ch = torch.full((M, N), 9.0, dtype=torch.float16).pin_memory()
    Ad = torch.empty_like(A, device=DEV)
    Bd = torch.empty_like(B, device=DEV)
    Cd = torch.empty((M, N), dtype=torch.float16, device=DEV)
    s = torch.cuda.Stream()
    g.gemm_f16_from_host(Ah, Bh, Ch, Ad, Bd, Cd, relu=True, stream=s)
    s.synchronize()
    assert g.check(stream=s) == g.GEMM_OK
    rows = sample_rows(M, seed=M)
    assert_close(Ch.numpy()[rows], oracle.gemm_f16(A, B, relu=True, rows=rows), f"from_host M={M}")
    assert not np.any(Ch.numpy() == np.float16(9.0))


@pytest.mark.parametrize("M,N,K", [(2500, 5000, 1000), (8192, 8192, 512), (700, 3000, 264)])
def test_from_host_ragged_shapes_bit_exact(g, M, N, K):
    # larger, ragged shapes through the host-buffer call: every element of C
    # comes down (no sentinel left), bit for bit on integer operands
    A, B = draw(M, N, K, "integer", seed=M + N)
    Ah, Bh = A.pin_memory(), B.pin_memory()
    Ch = torch.full((M, N), 9.5, dtype=torch.float16).pin_memory()
    Ad = torch.empty_like(A, device=DEV)
    Bd = torch.empty_like(B, device=DEV)
    Cd = torch.empty((M, N), dtype=torch.float16, device=DEV)
    g.gemm_f16_from_host(Ah, Bh, Ch, Ad, Bd, Cd, relu=False)
    torch.cuda.synchronize()
    assert g.check() == g.GEMM_OK
    got = Ch.numpy()
    assert not np.any(got.view(np.uint16) == np.float16(9.5).view(np.uint16))   # every block came down
    # integer operands: every partial sum is exact in fp32, one rounding to
    # fp16 as in the oracle, so the comparison is bit for bit
    rows = sorted(set(sample_rows(M, seed=N)) | {1023, 1024, 1279, 1280, 2047, 2048} & set(range(M)))
    ref = oracle.gemm_f16(A, B, relu=False, rows=rows)
    assert np.array_equal(got[rows].view(np.uint16), ref.view(np.uint16)), (M, N, K)
    # the device result equals the host copy
    assert np.array_equal(Cd.cpu().numpy().view(np.uint16), got.view(np.uint16))


def test_from_host_two_streams_in_flight(g):
    # The pattern of a caller streaming independent problems: steps alternate
    # between two streams, each with its own device buffers and host result,
    # and nothing is synchronised until the end, so one step's uploads run
    # while the previous step's GEMMs and downloads finish.  Every step's
    # result must be its own problem's, bit for bit (integer operands).
    M, N, K = 2304, 1024, 768
    steps = 4
    probs = [draw(M, N, K, "integer", seed=900 + i) for i in range(steps)]
    hosts = [(A.pin_memory(), B.pin_memory(), torch.full((M, N), 9.5, dtype=torch.float16).pin_memory())
             for A, B in probs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    devs = [(torch.empty((M, K), dtype=torch.float16, device=DEV), torch.empty((K, N), dtype=torch.float16, device=DEV),
             torch.empty((M, N), dtype=torch.float16, device=DEV)) for _ in range(2)]
    for i in range(steps):
        Ah, Bh, Ch = hosts[i]
        Ad, Bd, Cd = devs[i % 2]
        g.gemm_f16_from_host(Ah, Bh, Ch, Ad, Bd, Cd, relu=bool(i % 2), stream=streams[i % 2])
    for s in streams:
        s.synchronize()
        assert g.check(stream=s) == g.GEMM_OK
    for i, (A, B) in enumerate(probs):
        rows = sorted(set(sample_rows(M, seed=i)) | {0, 1023, 1024, 2303})
        ref = oracle.gemm_f16(A, B, relu=bool(i % 2), rows=rows)
        assert np.array_equal(hosts[i][2].numpy()[rows].view(np.uint16), ref.view(np.uint16)), i


# ---------------------------------------------------------------- argument errors (nothing launched)

def test_rejects_bad_buffers(g):
    M = N = K = 64
    A = torch.zeros((M, K), dtype=torch.float16, device=DEV)
    B = torch.zeros((K, N), dtype=torch.float16, device=DEV)
    C = torch.zeros((M, N), dtype=torch.float16, device=DEV)
    big = torch.zeros(M * N + 8, dtype=torch.float16, device=DEV)
    raw = g.gemm_f16_raw
    # misaligned (2-byte offset)
    assert raw(big.data_ptr() + 2, B.data_ptr(), C.data_ptr(), M, N, K, 1) == g.GEMM_ERR_ALIGNMENT
    # N or K not a multiple of 8
    assert raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, 60, 64, 1) == g.GEMM_ERR_ALIGNMENT
    assert raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, 64, 60, 1) == g.GEMM_ERR_ALIGNMENT
    # host memory
    host = torch.zeros((M, K), dtype=torch.float16)
    assert raw(host.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, 1) == g.GEMM_ERR_INVALID_ARG
    pinned = host.pin_memory()
    assert raw(pinned.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, 1) == g.GEMM_ERR_INVALID_ARG
    # NULL
    assert raw(0, B.data_ptr(), C.data_ptr(), M, N, K, 1) == g.GEMM_ERR_INVALID_ARG
    # C overlapping A
    assert raw(big.data_ptr(), B.data_ptr(), big.data_ptr() + 16, M, N, K, 1) == g.GEMM_ERR_INVALID_ARG
    # buffer smaller than its matrix (a 64x64 A claimed to be 1<<20 rows)
    assert raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), 1 << 20, N, K, 1) in (g.GEMM_ERR_INVALID_ARG,)
    torch.cuda.synchronize()
    assert g.check() == g.GEMM_OK


def test_no_split_flag_keeps_results_identical(g):
    # 1000^3 leaves a partly filled last wave in every configuration, so the
    # default schedule splits it along N; the flag keeps whole tiles.  Each
    # output is the same K-ordered fp32 sum either way.
    w = WORKLOADS["relu_ragged_1000"]
    A, B = draw_workload(w)
    ref = oracle.gemm_f16(A, B, relu=True)
    for cfg in configs(g):
        split = run(g, A, B, True, cfg)
        whole = run(g, A, B, True, cfg | g.GEMM_F16_NO_SPLIT)
        assert np.array_equal(split.view(np.uint16), whole.view(np.uint16)), cfg
        assert_close(whole, ref, f"{w.name} cfg {cfg} no-split")


def test_auto_choice_is_a_valid_config(g):
    for (M, N, K) in [(8192, 8192, 8192), (4096, 4096, 4096), (1024, 1024, 1024), (64, 64, 64), (16384, 512, 64)]:
        c = g.auto_config(M, N, K)
        assert c > 0 and g.config_name(c) is not None
        assert (c & ~(g.GEMM_F16_CONFIG_ID_MASK | g.GEMM_F16_NO_SPLIT | g.GEMM_F16_KSPLIT_MASK)) == 0


def test_auto_config_follows_the_tuned_table(g):
    # on a measured shape the wave-efficiency rescaling is 1, so the automatic
    # choice is the candidate with the highest measured throughput
    import re
    from dense_fp16_gemm_05_gb300 import build as gbuild
    with open(f"{gbuild.CSRC}/gemm_f16_tuned.inc") as f:
        text = f.read()
    cands = [int(x, 16) for x in re.search(r"kTunedCandidates\[[^\]]*\] = \{([^}]*)\}", text).group(1).split(",")]
    # candidates the automatic choice may take: no workspace K split
    def allowed(c):
        return g.config_cluster_k(c) or not (c & (g.GEMM_F16_KSPLIT_AUTO | g.GEMM_F16_KSPLIT_TAIL
                                                  | g.GEMM_F16_KSPLIT_MASK))
    for m in re.finditer(r"\{(\d+), (\d+), (\d+), \{([^}]*)\}\}", text):
        M, N, K = (int(m.group(i)) for i in (1, 2, 3))
        vals = [float(x.strip().rstrip("f")) for x in m.group(4).split(",")]
        best = max((v, -i, c) for i, (v, c) in enumerate(zip(vals, cands)) if allowed(c))[2]
        got = g.auto_config(M, N, K)
        if g.config_cluster_k(best):
            # the cluster size, resolved for this shape (at most the one measured)
            n = (got & g.GEMM_F16_KSPLIT_MASK) >> g.GEMM_F16_KSPLIT_SHIFT
            want = (best & g.GEMM_F16_KSPLIT_MASK) >> g.GEMM_F16_KSPLIT_SHIFT
            assert (got & g.GEMM_F16_CONFIG_ID_MASK) == (best & g.GEMM_F16_CONFIG_ID_MASK), (M, N, K, hex(got))
            assert n <= (want or 8), (M, N, K, hex(got))
        elif best & g.GEMM_F16_KSPLIT_AUTO:
            # the rule's slice count, resolved for this shape (whole tiles then)
            n = (got & g.GEMM_F16_KSPLIT_MASK) >> g.GEMM_F16_KSPLIT_SHIFT
            plain = best & ~g.GEMM_F16_KSPLIT_AUTO
            assert got == plain or (n >= 2 and got == plain | g.GEMM_F16_NO_SPLIT | g.ksplit(n)), (M, N, K, hex(got))
        else:
            assert got == best, (M, N, K, hex(got))
