"""Pins for the CPU oracle: checks against facts that do not come from it.

Each test ties one part of the oracle to something fixed independently:
numpy's binary16 conversions (exhaustive and on ties), closed forms of the
matrix product (identity, permutation, all-negative products), an int64
brute-force matmul on small integers, and the hand-derived cases in
``tests/golden/hand_cases.json``.  The last test checks that these pins are
sensitive: plausible mistakes (a dropped term, a transposed operand, a wrong
sign, ReLU after the cast on -0, a truncating cast) each fail at least one.

Definition followed: "Writing High-Performance Kernels in TileLang, from GEMM
to MLA" (atlascloud.ai), section "Let's write a GEMM" -- C = ReLU(A @ B) on
float16 operands with a float accumulator, ReLU on the accumulator, one cast
at write-back.
"""
from __future__ import annotations

import json
import os

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def bits(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x).view(np.uint16)


def int_matmul_f16(a_int: np.ndarray, b_int: np.ndarray, relu: bool) -> np.ndarray:
    """int64 brute force, then one correctly rounded conversion to binary16."""
    c = a_int.astype(np.int64) @ b_int.astype(np.int64)
    if relu:
        c = np.maximum(c, 0)
    with np.errstate(over="ignore"):
        return c.astype(np.float64).astype(np.float16)


# --------------------------------------------------------------------------
# Conversions, against numpy (exact decode; correctly rounded float64 -> half)
# --------------------------------------------------------------------------

def test_decode_all_binary16_patterns(oracle_mod):
    allbits = np.arange(65536, dtype=np.uint16)
    ours = oracle_mod.f16_to_f64(allbits)
    ref = allbits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # sign of zero is kept
    assert np.signbit(ours[0x8000]) and not np.signbit(ours[0x0000])


def test_encode_round_trips_every_pattern(oracle_mod):
    allbits = np.arange(65536, dtype=np.uint16)
    vals = allbits.view(np.float16).astype(np.float64)
    ok = ~np.isnan(vals)
    back = oracle_mod.f64_to_f16_bits(vals[ok])
    assert np.array_equal(back, allbits[ok])


def test_encode_ties_go_to_even(oracle_mod):
    # midpoints of every pair of adjacent finite positive binary16 values
    lo = np.arange(0x0000, 0x7bff, dtype=np.uint16)
    hi = lo + 1
    lv = lo.view(np.float16).astype(np.float64)
    hv = hi.view(np.float16).astype(np.float64)
    mid = (lv + hv) / 2.0  # exact in float64
    got = oracle_mod.f64_to_f16_bits(mid)
    want = np.where(lo % 2 == 0, lo, hi).astype(np.uint16)
    assert np.array_equal(got, want)
    # negative midpoints mirror
    got_neg = oracle_mod.f64_to_f16_bits(-mid)
    assert np.array_equal(got_neg, want | 0x8000)
    # one float64 ulp either side of each midpoint decides the direction
    below = np.nextafter(mid, 0.0)
    above = np.nextafter(mid, np.inf)
    assert np.array_equal(oracle_mod.f64_to_f16_bits(below), lo)
    assert np.array_equal(oracle_mod.f64_to_f16_bits(above), hi)


def test_encode_matches_numpy_on_random_values(oracle_mod):
    rng = np.random.default_rng(12345)
    parts = [
        rng.standard_normal(20000),                          # ordinary values
        rng.standard_normal(20000) * 2.0 ** -15,             # subnormal range
        rng.uniform(60000, 70000, 5000),                     # near overflow
        rng.standard_normal(5000) * 2.0 ** -26,              # below the smallest subnormal
        np.ldexp(rng.uniform(1, 2, 5000), rng.integers(-30, 20, 5000)),
    ]
    x = np.concatenate(parts)
    x = np.concatenate([x, -x])
    got = oracle_mod.f64_to_f16_bits(x)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def test_encode_special_values(oracle_mod):
    cases = [  # a list, not a dict: 0.0 and -0.0 are equal keys
        (0.0, 0x0000), (-0.0, 0x8000), (65504.0, 0x7BFF), (65519.99, 0x7BFF), (65520.0, 0x7C00),
        (1e6, 0x7C00), (-1e6, 0xFC00), (float("inf"), 0x7C00), (float("-inf"), 0xFC00),
        (2.0 ** -24, 0x0001), (2.0 ** -25, 0x0000), (1.5 * 2.0 ** -25, 0x0001),
        (3 * 2.0 ** -26, 0x0001), (2.0 ** -14, 0x0400), ((2.0 ** -14) * (1 - 2.0 ** -11), 0x0400),
    ]
    for v, want in cases:
        assert int(oracle_mod.f64_to_f16_bits([v])[0]) == want, v
    nan_bits = int(oracle_mod.f64_to_f16_bits([float("nan")])[0])
    assert (nan_bits & 0x7C00) == 0x7C00 and (nan_bits & 0x03FF) != 0


# --------------------------------------------------------------------------
# Whole GEMM: hand-derived cases
# --------------------------------------------------------------------------

def _load_hand_cases():
    with open(os.path.join(HERE, "golden", "hand_cases.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _load_hand_cases(), ids=lambda c: c["name"])
def test_hand_derived_cases(oracle_mod, case):
    def mat(rows):
        return np.array([[int(v, 16) for v in r] for r in rows], dtype=np.uint16)
    A, B, C = mat(case["A"]), mat(case["B"]), mat(case["C"])
    assert A.shape == (case["M"], case["K"]) and B.shape == (case["K"], case["N"])
    got = bits(oracle_mod.gemm_f16(A, B, relu=bool(case["relu"])))
    assert np.array_equal(got, C), (case["name"], [hex(v) for v in got.ravel()])


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------

def _normal_f16(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


@pytest.mark.parametrize("relu", [False, True])
def test_identity_reproduces_b(oracle_mod, relu):
    rng = np.random.default_rng(1)
    K, N = 37, 29
    B = _normal_f16(rng, (K, N))
    eye = np.eye(K, dtype=np.float16)
    C = oracle_mod.gemm_f16(eye, B, relu=relu)
    if relu:
        want = np.where(B > 0, B, np.float16(0.0)).astype(np.float16)
    else:
        want = B + np.float16(0.0)  # -0 entries of B become +0 (the sum starts at +0)
    assert np.array_equal(bits(C), bits(want))
    # and on the right: A @ I == A
    A = _normal_f16(rng, (N, K))
    C2 = oracle_mod.gemm_f16(A, eye, relu=False)
    assert np.array_equal(bits(C2), bits(A + np.float16(0.0)))


def test_permutations_move_rows_and_columns(oracle_mod):
    rng = np.random.default_rng(2)
    M, K, N = 23, 31, 19
    A = _normal_f16(rng, (M, K))
    B = _normal_f16(rng, (K, N))
    # P @ B permutes the rows of B
    perm = rng.permutation(K)
    P = np.zeros((K, K), dtype=np.float16)
    P[np.arange(K), perm] = 1
    assert np.array_equal(bits(oracle_mod.gemm_f16(P, B, relu=False)), bits(B[perm] + np.float16(0)))
    # A @ Q with Q[perm[j], j] = 1 picks column perm[j] of A
    perm2 = rng.permutation(K)[:N] if N <= K else None
    Q = np.zeros((K, N), dtype=np.float16)
    Q[perm2, np.arange(N)] = 1
    assert np.array_equal(bits(oracle_mod.gemm_f16(A, Q, relu=False)), bits(A[:, perm2] + np.float16(0)))


def test_all_negative_products(oracle_mod):
    rng = np.random.default_rng(3)
    M, K, N = 17, 40, 13
    a = rng.integers(1, 5, (M, K))       # positive
    b = -rng.integers(1, 5, (K, N))      # negative
    A, B = a.astype(np.float16), b.astype(np.float16)
    Crelu = oracle_mod.gemm_f16(A, B, relu=True)
    assert np.all(bits(Crelu) == 0x0000)                 # +0 everywhere, never -0
    Cplain = oracle_mod.gemm_f16(A, B, relu=False)
    assert np.array_equal(bits(Cplain), bits(int_matmul_f16(a, b, relu=False)))
    assert np.all(Cplain.astype(np.float64) < 0)


def test_k_zero_gives_plus_zero(oracle_mod):
    for relu in (False, True):
        C = oracle_mod.gemm_f16(np.zeros((5, 0), np.float16), np.zeros((0, 7), np.float16), relu=relu)
        assert C.shape == (5, 7) and np.all(bits(C) == 0)


def test_empty_m_or_n(oracle_mod):
    assert oracle_mod.gemm_f16(np.zeros((0, 4), np.float16), np.zeros((4, 3), np.float16), True).shape == (0, 3)
    assert oracle_mod.gemm_f16(np.zeros((2, 4), np.float16), np.zeros((4, 0), np.float16), True).shape == (2, 0)


def test_nan_and_inf_readings(oracle_mod):
    A = np.array([[np.nan, 1.0], [np.inf, 1.0], [-np.inf, 1.0]], dtype=np.float16)
    B = np.array([[1.0], [1.0]], dtype=np.float16)
    plain = oracle_mod.gemm_f16(A, B, relu=False).astype(np.float64).ravel()
    assert np.isnan(plain[0]) and plain[1] == np.inf and plain[2] == -np.inf
    relu = bits(oracle_mod.gemm_f16(A, B, relu=True)).ravel()
    assert list(relu) == [0x0000, 0x7C00, 0x0000]  # NaN -> +0, +inf kept, -inf -> +0


# --------------------------------------------------------------------------
# Brute force on small integers (every partial sum exact)
# --------------------------------------------------------------------------

SHAPES = [(1, 1, 1), (1, 17, 1), (17, 1, 1), (1, 1, 17), (3, 5, 7), (7, 3, 5), (8, 8, 8),
          (16, 9, 13), (17, 17, 17), (2, 64, 3), (64, 64, 64), (33, 65, 129)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("relu", [False, True])
def test_small_integers_bit_exact_vs_int64(oracle_mod, shape, relu):
    M, N, K = shape
    rng = np.random.default_rng(M * 10007 + N * 101 + K)
    a = rng.integers(-4, 5, (M, K))
    b = rng.integers(-4, 5, (K, N))
    got = oracle_mod.gemm_f16(a.astype(np.float16), b.astype(np.float16), relu=relu)
    assert np.array_equal(bits(got), bits(int_matmul_f16(a, b, relu)))


def test_large_integer_sums_round_like_numpy(oracle_mod):
    # sums beyond 2048 are not all representable: the single final rounding
    # must match numpy's correctly rounded int -> float16 conversion
    rng = np.random.default_rng(7)
    a = rng.integers(0, 64, (9, 300))
    b = rng.integers(0, 64, (300, 11))
    got = oracle_mod.gemm_f16(a.astype(np.float16), b.astype(np.float16), relu=False)
    assert np.array_equal(bits(got), bits(int_matmul_f16(a, b, False)))


# --------------------------------------------------------------------------
# Row selection and the ReLU invariant
# --------------------------------------------------------------------------

def test_row_selection_matches_full(oracle_mod):
    rng = np.random.default_rng(5)
    A = _normal_f16(rng, (50, 70))
    B = _normal_f16(rng, (70, 40))
    full = oracle_mod.gemm_f16(A, B, relu=True)
    rows = [49, 0, 17, 17, 3]
    part = oracle_mod.gemm_f16(A, B, relu=True, rows=rows)
    assert np.array_equal(bits(part), bits(full[rows]))


def test_relu_is_max_with_plus_zero(oracle_mod):
    rng = np.random.default_rng(6)
    A = _normal_f16(rng, (40, 64))
    B = _normal_f16(rng, (64, 48))
    plain = oracle_mod.gemm_f16(A, B, relu=False)
    relu = oracle_mod.gemm_f16(A, B, relu=True)
    want = np.where(plain.astype(np.float64) > 0, plain, np.float16(0.0)).astype(np.float16)
    assert np.array_equal(bits(relu), bits(want))


def test_normal_inputs_within_fp64_reference(oracle_mod):
    # an independent float64 matmul (numpy) rounded once must agree exactly
    # except where the float64 sums differ in rounding order -- allow 1 ulp
    rng = np.random.default_rng(8)
    A = _normal_f16(rng, (64, 256))
    B = _normal_f16(rng, (256, 96))
    got = oracle_mod.gemm_f16(A, B, relu=False).astype(np.float64)
    ref = (A.astype(np.float64) @ B.astype(np.float64)).astype(np.float16).astype(np.float64)
    ulp = np.spacing(np.abs(ref).astype(np.float16)).astype(np.float64)
    assert np.all(np.abs(got - ref) <= ulp)
    assert np.mean(got == ref) > 0.999


# --------------------------------------------------------------------------
# Sensitivity: plausible mistakes must each fail a pin
# --------------------------------------------------------------------------

def test_pins_catch_planted_mistakes(oracle_mod):
    """Plants mistakes in a copy of the oracle's arithmetic (on the CPU, in
    Python) and checks that the pin data used above rejects every one."""
    rng = np.random.default_rng(9)
    a = rng.integers(-4, 5, (7, 5))
    b = rng.integers(-4, 5, (5, 6))
    A, B = a.astype(np.float16), b.astype(np.float16)
    truth = bits(int_matmul_f16(a, b, relu=True))
    hand = {c["name"]: c for c in _load_hand_cases()}

    def run(mutant, A_, B_, relu):
        a64 = A_.astype(np.float64)
        b64 = B_.astype(np.float64)
        return mutant(a64, b64, relu)

    def correct(a64, b64, relu):
        acc = np.zeros((a64.shape[0], b64.shape[1]))
        for k in range(a64.shape[1]):
            acc = acc + np.outer(a64[:, k], b64[k, :])
        if relu:
            acc = np.where(acc > 0, acc, 0.0)
        return acc.astype(np.float16)

    def dropped_last_term(a64, b64, relu):
        return correct(a64[:, :-1], b64[:-1, :], relu)

    def transposed_b(a64, b64, relu):
        # reads B's memory as if it were (N,K) row-major: B[j*K + k] for B[k*N + j]
        K_, N_ = b64.shape
        return correct(a64, b64.ravel().reshape(N_, K_).T, relu)

    def transposed_a(a64, b64, relu):
        M_, K_ = a64.shape
        return correct(a64.ravel().reshape(K_, M_).T, b64, relu)

    def wrong_sign(a64, b64, relu):
        return correct(a64, -b64, relu)

    def relu_after_cast_keeps_minus_zero(a64, b64, relu):
        acc = a64 @ b64
        c = acc.astype(np.float16)
        if relu:
            c = np.where(c < 0, np.float16(-0.0), c).astype(np.float16)
        return c

    def truncating_cast(a64, b64, relu):
        acc = a64 @ b64
        if relu:
            acc = np.where(acc > 0, acc, 0.0)
        c = acc.astype(np.float16)
        over = np.abs(c.astype(np.float64)) > np.abs(acc)
        return np.where(over, np.nextafter(c, np.float16(0)), c).astype(np.float16)

    def pins_pass(mutant):
        if not np.array_equal(bits(run(mutant, A, B, True)), truth):
            return False
        for name in ("tie_rounds_down_to_even", "tie_rounds_up_to_even", "relu_of_negative_sum_is_plus_zero",
                     "rectangular_2x3_times_3x2", "just_above_tie_with_subnormal_term"):
            c = hand[name]
            mat = lambda rows: np.array([[int(v, 16) for v in r] for r in rows], dtype=np.uint16).view(np.float16)
            got = bits(run(mutant, mat(c["A"]), mat(c["B"]), bool(c["relu"])))
            if not np.array_equal(got, mat(c["C"]).view(np.uint16)):
                return False
        return True

    assert pins_pass(correct)
    for m in (dropped_last_term, transposed_b, transposed_a, wrong_sign, relu_after_cast_keeps_minus_zero, truncating_cast):
        assert not pins_pass(m), m.__name__


# --------------------------------------------------------------------------
# ReLU gradient and transposed operands
# --------------------------------------------------------------------------

def test_relu_backward_hand_cases(oracle_mod):
    with open(os.path.join(HERE, "golden", "relu_backward_cases.json")) as f:
        case = json.load(f)
    C = np.array([int(v, 16) for v in case["C"]], dtype=np.uint16)
    dC = np.array([int(v, 16) for v in case["dC"]], dtype=np.uint16)
    want = np.array([int(v, 16) for v in case["dZ"]], dtype=np.uint16)
    got = bits(oracle_mod.relu_backward(dC, C))
    assert np.array_equal(got, want), [hex(v) for v in got]


def test_relu_backward_mask_matches_forward_sign(oracle_mod):
    # where the forward output is positive the gradient passes, elsewhere +0
    rng = np.random.default_rng(10)
    a = rng.integers(-4, 5, (12, 20))
    b = rng.integers(-4, 5, (20, 9))
    C = oracle_mod.gemm_f16(a.astype(np.float16), b.astype(np.float16), relu=True)
    dC = rng.integers(-8, 9, C.shape).astype(np.float16)
    dZ = oracle_mod.relu_backward(dC, C)
    z = a @ b   # exact int64 pre-activation
    assert np.array_equal(bits(dZ), bits(np.where(z > 0, dC, np.float16(0)).astype(np.float16)))


@pytest.mark.parametrize("transa,transb", [(False, True), (True, False), (True, True)])
def test_transposed_layouts_vs_int64(oracle_mod, transa, transb):
    rng = np.random.default_rng(11 + 2 * transa + transb)
    M, N, K = 13, 17, 29
    a = rng.integers(-4, 5, (M, K))
    b = rng.integers(-4, 5, (K, N))
    A_st = a.T.copy() if transa else a
    B_st = b.T.copy() if transb else b
    got = oracle_mod.gemm_f16_t(A_st.astype(np.float16), B_st.astype(np.float16), relu=False,
                                transa=transa, transb=transb)
    assert np.array_equal(bits(got), bits(int_matmul_f16(a, b, relu=False)))
