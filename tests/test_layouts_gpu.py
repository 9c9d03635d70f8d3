"""GPU parity of the transposed operand layouts, the ReLU gradient kernel and
the autograd wrapper, against the CPU oracle.

Layouts follow the transpose_A / transpose_B options of the tile GEMM
("Writing High-Performance Kernels in TileLang, from GEMM to MLA", section
"Let's write a GEMM"); the backward pair dA = dC @ B^T, dB = A^T @ dC is the
autograd wrapper of the TileLang-MUSA lesson (section 6).  Tolerance as for
the forward kernel: |gpu - ref| <= 2e-2 + 2e-3 |ref|; bit-exact on
integer-valued inputs and for the (integer-only) ReLU mask.
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
LAYOUTS = [(False, True), (True, False), (True, True), (False, False)]


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from dense_fp16_gemm_05_gb300 import build as gbuild
    gbuild.build()
    from dense_fp16_gemm_05_gb300 import gemm_f16
    gemm_f16.lib()
    return gemm_f16


def layout_configs(g):
    return [c for c in range(1, g.num_configs() + 1) if g.config_layouts(c) == 0xF]


def stored(X, trans):
    return X.t().contiguous() if trans else X


def assert_close(got, ref, what):
    got64 = got.astype(np.float64)
    ref64 = ref.astype(np.float64)
    err = np.abs(got64 - ref64)
    bad = err > ATOL + RTOL * np.abs(ref64)
    assert not np.isnan(got64).any(), what
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside tolerance, max err {err.max():.4g}"


@pytest.mark.parametrize("transa,transb", LAYOUTS)
@pytest.mark.parametrize("M,N,K", [(1000, 1000, 1000), (264, 136, 200), (128, 512, 64), (520, 264, 72)])
def test_transposed_layouts_match_oracle(g, transa, transb, M, N, K):
    A, B = draw(M, N, K, "normal", seed=M + 3 * N + 7 * K)    # op(A) (M,K), op(B) (K,N)
    A_st, B_st = stored(A, transa), stored(B, transb)
    ref = oracle.gemm_f16_t(A_st, B_st, relu=True, transa=transa, transb=transb)
    for cfg in layout_configs(g):
        C = g.gemm_f16_t(A_st.to(DEV), B_st.to(DEV), transa=transa, transb=transb, relu=True, config=cfg)
        assert g.check() == g.GEMM_OK
        assert_close(C.cpu().numpy(), ref, f"layout ({transa},{transb}) {M}x{N}x{K} cfg {cfg}")


@pytest.mark.parametrize("transa,transb", LAYOUTS)
def test_transposed_layouts_integers_bit_exact(g, transa, transb):
    A, B = draw(64, 64, 64, "integer", seed=41)
    A_st, B_st = stored(A, transa), stored(B, transb)
    ref = oracle.gemm_f16_t(A_st, B_st, relu=True, transa=transa, transb=transb)
    for cfg in layout_configs(g):
        C = g.gemm_f16_t(A_st.to(DEV), B_st.to(DEV), transa=transa, transb=transb, relu=True, config=cfg)
        assert np.array_equal(C.cpu().numpy().view(np.uint16), ref.view(np.uint16)), cfg


def test_transposed_large_sampled(g):
    # the backward shapes of the 8192^3 forward, in the automatic configuration
    n = 8192
    A, B = draw(n, n, n, "normal_scaled", seed=5)
    rows = [0, 1, 255, 256, 4095, 8191, 1234, 7777]
    for transa, transb in [(False, True), (True, False)]:
        A_st, B_st = stored(A, transa), stored(B, transb)
        C = g.gemm_f16_t(A_st.to(DEV), B_st.to(DEV), transa=transa, transb=transb, relu=False)
        assert g.check() == g.GEMM_OK
        ref = oracle.gemm_f16_t(A_st, B_st, relu=False, transa=transa, transb=transb, rows=rows)
        assert_close(C.cpu().numpy()[rows], ref, f"8192^3 layout ({transa},{transb})")


def test_layout_alignment_rules(g):
    # transposed A needs M % 8 == 0 (its row pitch); plain A does not
    A = torch.zeros((64, 60), dtype=torch.float16, device=DEV)      # stored (K=64, M=60)
    B = torch.zeros((64, 64), dtype=torch.float16, device=DEV)
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16_t(A, B, transa=True)
    assert e.value.status == g.GEMM_ERR_ALIGNMENT
    # configurations without transposed kernels refuse the layout
    for cfg in range(1, g.num_configs() + 1):
        if g.config_layouts(cfg) != 0xF:
            with pytest.raises(g.GemmError):
                g.gemm_f16_t(B, B, transb=True, config=cfg)


def test_relu_backward_bit_exact(g):
    rng = np.random.default_rng(12)
    for n in (1, 7, 8, 9, 4096 * 8 + 5, 3_000_001):
        C = rng.integers(0, 65536, n, dtype=np.uint16)     # every class of binary16 value
        dC = rng.integers(0, 65536, n, dtype=np.uint16)
        ref = oracle.relu_backward(dC, C).view(np.uint16)
        Ct = torch.from_numpy(C.view(np.float16)).to(DEV)
        dCt = torch.from_numpy(dC.view(np.float16)).to(DEV)
        got = g.relu_backward(dCt, Ct)
        assert g.check() == g.GEMM_OK
        assert np.array_equal(got.cpu().numpy().view(np.uint16), ref), n
        # misaligned views take the scalar path
        if n > 9:
            got2 = g.relu_backward(dCt[1:], Ct[1:])
            assert np.array_equal(got2.cpu().numpy().view(np.uint16), ref[1:]), n
    # in place over dC
    C = rng.integers(0, 65536, 1000, dtype=np.uint16)
    dC = rng.integers(0, 65536, 1000, dtype=np.uint16)
    ref = oracle.relu_backward(dC, C).view(np.uint16)
    dCt = torch.from_numpy(dC.view(np.float16)).to(DEV)
    g.relu_backward(dCt, torch.from_numpy(C.view(np.float16)).to(DEV), dZ=dCt)
    assert np.array_equal(dCt.cpu().numpy().view(np.uint16), ref)


@pytest.mark.parametrize("relu", [True, False])
def test_autograd_integer_bit_exact(g, relu):
    from dense_fp16_gemm_05_gb300.autograd import GemmF16Function
    M = N = K = 64
    A, B = draw(M, N, K, "integer", seed=51)
    rng = np.random.default_rng(52)
    G = rng.integers(-4, 5, (M, N)).astype(np.float16)
    Ad = A.to(DEV).requires_grad_(True)
    Bd = B.to(DEV).requires_grad_(True)
    C = GemmF16Function.apply(Ad, Bd, relu)
    C.backward(torch.from_numpy(G).to(DEV))
    # oracle: forward, mask, then the backward pair with transposed operands
    C_ref = oracle.gemm_f16(A, B, relu=relu)
    dZ = oracle.relu_backward(G, C_ref) if relu else G
    dA_ref = oracle.gemm_f16_t(dZ, B, relu=False, transb=True)
    dB_ref = oracle.gemm_f16_t(A, dZ, relu=False, transa=True)
    assert np.array_equal(C.detach().cpu().numpy().view(np.uint16), C_ref.view(np.uint16))
    assert np.array_equal(Ad.grad.cpu().numpy().astype(np.float64), dA_ref.astype(np.float64))
    assert np.array_equal(Bd.grad.cpu().numpy().astype(np.float64), dB_ref.astype(np.float64))


def test_autograd_plain_normal_values(g):
    from dense_fp16_gemm_05_gb300.autograd import gemm
    M, N, K = 512, 384, 256
    A, B = draw(M, N, K, "normal", seed=53)
    rng = np.random.default_rng(55)
    Gn = rng.standard_normal((M, N)).astype(np.float16)
    Ad = A.to(DEV).requires_grad_(True)
    Bd = B.to(DEV).requires_grad_(True)
    gemm(Ad, Bd).backward(torch.from_numpy(Gn).to(DEV))
    assert_close(Ad.grad.cpu().numpy(), oracle.gemm_f16_t(Gn, B, relu=False, transb=True), "dA")
    assert_close(Bd.grad.cpu().numpy(), oracle.gemm_f16_t(A, Gn, relu=False, transa=True), "dB")


def test_calls_from_a_fresh_thread(g):
    # the library must work on a thread whose first CUDA call is its own
    import threading
    A, B = draw(256, 256, 128, "normal", seed=61)
    Ad, Bd = A.to(DEV), B.to(DEV)
    out = {}

    def work():
        try:
            C = g.gemm_f16(Ad, Bd, relu=True)
            dZ = g.relu_backward(C, C)
            torch.cuda.synchronize(DEV)
            out["C"] = C.cpu().numpy()
            out["dZ"] = dZ.cpu().numpy()
        except Exception as e:      # reported below
            out["err"] = e

    t = threading.Thread(target=work)
    t.start()
    t.join()
    assert "err" not in out, out.get("err")
    assert_close(out["C"], oracle.gemm_f16(A, B, relu=True), "fresh thread")
