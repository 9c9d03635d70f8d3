"""Pins for the FP8 block-scaled oracle (CPU only).

What the oracle computes is the plainest reading of the FP8 block-scaled
linear layer of the TileLang-MUSA lesson (7yue.com, section 8.2,
fp8_block_scaled_linear(x, w_fp8, scale_w, block=128)) with the per-block
scaling the nxmr.cn TileLang article (section 7) names:

    C[i,j] = f16( R( sum_b SA[i,b] * SW[j/block, b] * sum_{k in block b} A[i,k] W[j,k] ) )

with A (M,K) and W (N,K) in OCP FP8 E4M3.  The pins tie it to facts that do
not come from the oracle: torch's E4M3 decoding on all 256 codes, hand-derived
cases (tests/golden/fp8_block_scaled_cases.json), exact rational arithmetic
(Python Fractions) on integer operands with power-of-two scales, and the
reductions of the definition at block = 1 and block >= K.  Planted mistakes
in a restatement (a shifted block index, transposed weight scales, a lost
partial block, scales added instead of multiplied) each fail.
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))


def e4m3_codes(values) -> np.ndarray:
    """E4M3 codes of exactly representable values (torch's encoder)."""
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def exact_result(a_int, sa, w_int, sw, block, relu):
    """The definition in exact rational arithmetic: integer-valued operands,
    scales that are exact binary fractions; returns float16 bits."""
    M, K = a_int.shape
    N = w_int.shape[0]
    KB = -(-K // block)
    out = np.empty((M, N), dtype=np.float16)
    for i in range(M):
        for j in range(N):
            acc = Fraction(0)
            for b in range(KB):
                p = sum(int(a_int[i, k]) * int(w_int[j, k]) for k in range(b * block, min(K, (b + 1) * block)))
                acc += Fraction(float(sa[i, b])) * Fraction(float(sw[j // block, b])) * p
            if relu and acc <= 0:
                acc = Fraction(0)
            # exact in float64 (small integers times powers of two), then one
            # correctly rounded conversion to binary16
            out[i, j] = np.float16(float(acc))
    return out.view(np.uint16)


def int_problem(rng, M, N, K, block, lo=-4, hi=4, emin=-3, emax=3):
    a = rng.integers(lo, hi + 1, (M, K))
    w = rng.integers(lo, hi + 1, (N, K))
    KB, NB = -(-K // block), -(-N // block)
    sa = np.ldexp(1.0, rng.integers(emin, emax + 1, (M, KB))).astype(np.float32)
    sw = np.ldexp(1.0, rng.integers(emin, emax + 1, (NB, KB))).astype(np.float32)
    return a, w, sa, sw


# --------------------------------------------------------------------------
# E4M3 decoding
# --------------------------------------------------------------------------

def test_e4m3_decode_all_codes_match_torch(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle_mod.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_e4m3_named_values(oracle_mod):
    named = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x30: 0.5, 0x38: 1.0,
             0x40: 2.0, 0x44: 3.0, 0x7E: 448.0, 0xBC: -1.5, 0xFE: -448.0}
    for code, v in named.items():
        assert oracle_mod.e4m3_to_f64([code])[0] == v, hex(code)
    assert np.signbit(oracle_mod.e4m3_to_f64([0x80])[0])
    assert np.isnan(oracle_mod.e4m3_to_f64([0x7F, 0xFF])).all()


# --------------------------------------------------------------------------
# Hand-derived cases
# --------------------------------------------------------------------------

def _hand_cases():
    with open(os.path.join(HERE, "golden", "fp8_block_scaled_cases.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _hand_cases(), ids=lambda c: c["name"])
def test_hand_cases(oracle_mod, case):
    A = np.array(case["A"], dtype=np.uint8)
    W = np.array(case["W"], dtype=np.uint8)
    SA = np.array(case["SA"], dtype=np.float32)
    SW = np.array(case["SW"], dtype=np.float32)
    got = oracle_mod.gemm_fp8_block_scaled(A, SA, W, SW, relu=bool(case["relu"]), block=case["block"])
    assert np.array_equal(got.view(np.uint16), np.array(case["C_bits"], dtype=np.uint16))


# --------------------------------------------------------------------------
# Exact arithmetic, closed forms
# --------------------------------------------------------------------------

@pytest.mark.parametrize("M,N,K,block", [(3, 5, 7, 128), (4, 6, 300, 128), (5, 200, 260, 128),
                                         (2, 3, 9, 4), (6, 7, 33, 8)])
@pytest.mark.parametrize("relu", [True, False])
def test_integer_operands_power_of_two_scales_exact(oracle_mod, M, N, K, block, relu):
    rng = np.random.default_rng(M * 1000 + N * 10 + K)
    a, w, sa, sw = int_problem(rng, M, N, K, block)
    got = oracle_mod.gemm_fp8_block_scaled(e4m3_codes(a), sa, e4m3_codes(w), sw, relu=relu, block=block)
    assert np.array_equal(got.view(np.uint16), exact_result(a, sa, w, sw, block, relu))


def test_unit_scales_reduce_to_the_plain_product(oracle_mod):
    # all scales 1: C = f16(R(A @ W^T)), an int64 matmul here
    rng = np.random.default_rng(3)
    a = rng.integers(-4, 5, (9, 300))
    w = rng.integers(-4, 5, (11, 300))
    sa = np.ones((9, 3), dtype=np.float32)
    sw = np.ones((1, 3), dtype=np.float32)
    got = oracle_mod.gemm_fp8_block_scaled(e4m3_codes(a), sa, e4m3_codes(w), sw, relu=False)
    ref = (a.astype(np.int64) @ w.astype(np.int64).T).astype(np.float16)
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))


def test_one_block_covering_k_scales_the_whole_product(oracle_mod):
    # block >= K: C[i,j] = SA[i,0] * SW[j/block,0] * (A @ W^T)[i,j]
    rng = np.random.default_rng(4)
    a = rng.integers(-3, 4, (4, 20))
    w = rng.integers(-3, 4, (5, 20))
    sa = np.array([[0.5], [2.0], [0.25], [4.0]], dtype=np.float32)
    sw = np.array([[8.0]], dtype=np.float32)
    got = oracle_mod.gemm_fp8_block_scaled(e4m3_codes(a), sa, e4m3_codes(w), sw, relu=False, block=64)
    ref = (sa.astype(np.float64) * 8.0 * (a @ w.T)).astype(np.float16)
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))


def test_block_one_gives_per_element_scales(oracle_mod):
    # block = 1: C[i,j] = sum_k SA[i,k] SW[j,k] A[i,k] W[j,k]
    rng = np.random.default_rng(5)
    a, w, sa, sw = int_problem(rng, 3, 4, 6, 1)
    got = oracle_mod.gemm_fp8_block_scaled(e4m3_codes(a), sa, e4m3_codes(w), sw, relu=False, block=1)
    ref = np.einsum("ik,jk,ik,jk->ij", sa.astype(np.float64), sw.astype(np.float64), a, w).astype(np.float16)
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))


def test_row_selection_matches_full_result(oracle_mod):
    rng = np.random.default_rng(6)
    a, w, sa, sw = int_problem(rng, 12, 9, 140, 128)
    full = oracle_mod.gemm_fp8_block_scaled(e4m3_codes(a), sa, e4m3_codes(w), sw, relu=True)
    rows = [11, 0, 5, 5]
    part = oracle_mod.gemm_fp8_block_scaled(e4m3_codes(a), sa, e4m3_codes(w), sw, relu=True, rows=rows)
    assert np.array_equal(part.view(np.uint16), full.view(np.uint16)[rows])


def test_shape_checks(oracle_mod):
    a = np.zeros((2, 10), np.uint8)
    with pytest.raises(ValueError):
        oracle_mod.gemm_fp8_block_scaled(a, np.ones((2, 2), np.float32), a, np.ones((1, 1), np.float32), True)


# --------------------------------------------------------------------------
# Sensitivity: plausible mistakes must fail the exact pin data
# --------------------------------------------------------------------------

def _restated(a, sa, w, sw, block, relu, mistake=None):
    M, K = a.shape
    N = w.shape[0]
    KB = -(-K // block)
    out = np.empty((M, N), dtype=np.float16)
    for i in range(M):
        for j in range(N):
            acc = 0.0
            for b in range(KB):
                ks = range(b * block, min(K, (b + 1) * block))
                if mistake == "drop_partial_block" and len(ks) < block:
                    continue
                p = float(sum(int(a[i, k]) * int(w[j, k]) for k in ks))
                s_a = float(sa[i, min(b + 1, KB - 1)]) if mistake == "shifted_block" else float(sa[i, b])
                if mistake == "transposed_weight_scales":
                    s_w = float(sw[b % sw.shape[0], (j // block) % sw.shape[1]])
                elif mistake == "weight_scale_by_row":
                    s_w = float(sw[(i // block) % sw.shape[0], b])
                else:
                    s_w = float(sw[j // block, b])
                acc += (s_a + s_w) * p if mistake == "scales_added" else s_a * s_w * p
            if relu and acc <= 0:
                acc = 0.0
            out[i, j] = np.float16(acc)
    return out.view(np.uint16)


@pytest.mark.parametrize("mistake", ["shifted_block", "transposed_weight_scales", "weight_scale_by_row",
                                     "drop_partial_block", "scales_added"])
def test_pins_catch_planted_mistakes(oracle_mod, mistake):
    rng = np.random.default_rng(11)
    a, w, sa, sw = int_problem(rng, 5, 200, 260, 128)     # 3 K blocks (last partial), 2 N blocks (last partial)
    truth = exact_result(a, sa, w, sw, 128, relu=False)
    assert np.array_equal(_restated(a, sa, w, sw, 128, False), truth)          # the harness itself is right
    assert not np.array_equal(_restated(a, sa, w, sw, 128, False, mistake), truth)
    got = oracle_mod.gemm_fp8_block_scaled(e4m3_codes(a), sa, e4m3_codes(w), sw, relu=False)
    assert np.array_equal(got.view(np.uint16), truth)


def test_fp8_input_recipes(oracle_mod):
    from dense_fp16_gemm_05_gb300.inputs import draw_fp8_block_scaled
    A, SA, W, SW = draw_fp8_block_scaled(70, 150, 260, "integer", 2)
    assert A.shape == (70, 260) and SA.shape == (70, 3) and W.shape == (150, 260) and SW.shape == (2, 3)
    a = oracle_mod.e4m3_to_f64(A.numpy())
    assert np.array_equal(a, np.round(a)) and np.abs(a).max() <= 4
    m, e = np.frexp(SA.numpy())
    assert np.all(m == 0.5)                               # powers of two
    A, SA, W, SW = draw_fp8_block_scaled(70, 150, 260, "normal", 3)
    w = oracle_mod.e4m3_to_f64(W.numpy())
    assert np.isfinite(w).all() and np.abs(w).max() <= 448
    # every block reaches the top code magnitude (scale = block max / 448)
    blk = np.abs(w[:128, :128])
    assert blk.max() == 448.0


# --------------------------------------------------------------------------
# Power-of-two scales given as E8M0 bytes (the block-scaled MMA's scale type)
# --------------------------------------------------------------------------

def _mx_golden():
    with open(os.path.join(HERE, "golden", "mxfp8_cases.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("entry", _mx_golden()["e8m0"], ids=lambda e: str(e["code"]))
def test_e8m0_named_values(oracle_mod, entry):
    got = oracle_mod.e8m0_to_f32(np.array([entry["code"]], dtype=np.uint8))[0]
    if entry["value"] == "nan":
        assert np.isnan(got)
    else:
        assert got == np.float32(entry["value"]) and got.dtype == np.float32


def test_e8m0_codes_are_consecutive_powers_of_two(oracle_mod):
    # each code doubles the one below it, from 2^-127 at code 0 (exact values)
    v = oracle_mod.e8m0_to_f32(np.arange(255, dtype=np.uint8)).astype(np.float64)
    assert np.array_equal(v[1:] / v[:-1], np.full(254, 2.0))
    assert v[0] == 2.0 ** -127 and v[127] == 1.0


def _runs_to_codes(runs):
    return np.array([[c for c, n in row for _ in range(n)] for row in runs], dtype=np.uint8)


@pytest.mark.parametrize("case", _mx_golden()["cases"], ids=lambda c: c["name"])
def test_mx_hand_cases(oracle_mod, case):
    A, W = _runs_to_codes(case["A_runs"]), _runs_to_codes(case["W_runs"])
    assert A.shape == (case["M"], case["K"]) and W.shape == (case["N"], case["K"])
    SA, SW = np.array(case["SA"], dtype=np.uint8), np.array(case["SW"], dtype=np.uint8)
    got = oracle_mod.gemm_mxfp8_block_scaled(A, SA, W, SW, relu=bool(case["relu"]))
    assert np.array_equal(got.view(np.uint16), np.array(case["C_bits"], dtype=np.uint16))


@pytest.mark.parametrize("relu", [True, False])
def test_mx_integer_operands_exact(oracle_mod, relu):
    # E8M0 exponents around the bias: the exact rational result, bit for bit
    rng = np.random.default_rng(21)
    M, N, K = 4, 200, 300
    a, w, _, _ = int_problem(rng, M, N, K, 128)
    ea = rng.integers(124, 131, (M, 3)).astype(np.uint8)
    ew = rng.integers(124, 131, (2, 3)).astype(np.uint8)
    sa = np.ldexp(1.0, ea.astype(np.int64) - 127).astype(np.float32)
    sw = np.ldexp(1.0, ew.astype(np.int64) - 127).astype(np.float32)
    got = oracle_mod.gemm_mxfp8_block_scaled(e4m3_codes(a), ea, e4m3_codes(w), ew, relu=relu)
    assert np.array_equal(got.view(np.uint16), exact_result(a, sa, w, sw, 128, relu))


def test_mx_pins_catch_an_off_by_one_bias(oracle_mod):
    # a decoder with bias 128 (or 126) would halve (double) every scale: the
    # first hand case then comes out 384 (1536) instead of 768
    case = _mx_golden()["cases"][0]
    A, W = _runs_to_codes(case["A_runs"]), _runs_to_codes(case["W_runs"])
    SA, SW = np.array(case["SA"], dtype=np.uint8), np.array(case["SW"], dtype=np.uint8)
    for bias in (126, 128):
        sa = np.ldexp(1.0, SA.astype(np.int64) - bias).astype(np.float32)
        sw = np.ldexp(1.0, SW.astype(np.int64) - bias).astype(np.float32)
        wrong = oracle_mod.gemm_fp8_block_scaled(A, sa, W, sw, relu=True)
        assert not np.array_equal(wrong.view(np.uint16), np.array(case["C_bits"], dtype=np.uint16))


def test_mx_input_recipes(oracle_mod):
    from dense_fp16_gemm_05_gb300.inputs import draw_mxfp8_block_scaled
    A, SA, W, SW = draw_mxfp8_block_scaled(70, 150, 260, "normal", 3)
    assert SA.dtype == torch.uint8 and SA.shape == (70, 3) and SW.shape == (2, 3)
    w = oracle_mod.e4m3_to_f64(W.numpy())
    assert np.isfinite(w).all() and np.abs(w).max() <= 448
    # a power-of-two scale rounded up: each block's largest code is in (224, 448]
    blk = np.abs(w[:128, :128])
    assert 224 < blk.max() <= 448
    A, SA, W, SW = draw_mxfp8_block_scaled(70, 150, 260, "integer", 2)
    a = oracle_mod.e4m3_to_f64(A.numpy())
    assert np.array_equal(a, np.round(a)) and np.abs(a).max() <= 4
    assert SA.numpy().min() >= 124 and SA.numpy().max() <= 130
