"""Pins for the attention-forward oracle (CPU only).

The oracle writes out the plain definition of what the FlashAttention loop
of the pages computes (TileLang-MUSA lesson, 7yue.com, section 5; "Writing
High-Performance Kernels in TileLang, from GEMM to MLA", the FlashAttention
loop of the MLA section): per (batch, head, query row i),

    O[i] = sum_j softmax_j(sm_scale * Q[i] . K[j]) V[j],  j < seq (j <= i if causal)

in fp64, rounded once to fp16.  Pins that do not restate that formula:
closed forms (zero queries give the mean of the value rows, exactly rounded;
one key gives that value row; a causal first row is V[0]; a score gap of 40
saturates the softmax), hand-derived cases (tests/golden/attention_cases.json),
invariants (a joint permutation of keys and values, moving a factor 2
between Q and sm_scale), and planted mistakes in a restatement (no max
subtraction, an off-by-one causal boundary, keys and values mismatched, the
softmax taken over queries, sm_scale dropped) each failing.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def f16_round_exact(x: Fraction) -> np.uint16:
    """Binary16 bits of the exact rational x, rounded to nearest, ties to even."""
    lo = np.float16(float(x))
    cands = {lo, np.nextafter(lo, np.float16(np.inf)), np.nextafter(lo, np.float16(-np.inf))}
    best = None
    for c in cands:
        if not np.isfinite(c):
            continue
        d = abs(Fraction(float(c)) - x)
        key = (d, int(np.array(c).view(np.uint16)) & 1)   # ties: even significand first
        if best is None or key < best[0]:
            best = (key, c)
    return np.array(best[1], dtype=np.float16).view(np.uint16)


def ulp_diff(a, b):
    ai = a.view(np.uint16).astype(np.int32)
    bi = b.view(np.uint16).astype(np.int32)
    ai = np.where(ai & 0x8000, -(ai & 0x7FFF), ai)
    bi = np.where(bi & 0x8000, -(bi & 0x7FFF), bi)
    return np.abs(ai - bi)


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_the_mean_of_the_values(oracle_mod, causal):
    rng = np.random.default_rng(1)
    S, D = 7, 5
    Q = np.zeros((1, 1, S, D), np.float16)
    K = rng.standard_normal((1, 1, S, D)).astype(np.float16)
    V = rng.standard_normal((1, 1, S, D)).astype(np.float16)
    got = oracle_mod.attention_fwd(Q, K, V, sm_scale=0.3, causal=causal)[0, 0]
    for i in range(S):
        n = i + 1 if causal else S
        for d in range(D):
            exact = sum(Fraction(float(V[0, 0, j, d])) for j in range(n)) / n
            assert got[i, d].view(np.uint16) == f16_round_exact(exact), (i, d)


def test_single_key_returns_its_value(oracle_mod):
    rng = np.random.default_rng(2)
    Q, K, V = (rng.standard_normal((2, 3, 1, 8)).astype(np.float16) for _ in range(3))
    for causal in (False, True):
        got = oracle_mod.attention_fwd(Q, K, V, sm_scale=1.0, causal=causal)
        assert np.array_equal(got.view(np.uint16), V.view(np.uint16))


def test_causal_first_row_is_the_first_value(oracle_mod):
    rng = np.random.default_rng(3)
    Q, K, V = (rng.standard_normal((1, 2, 9, 16)).astype(np.float16) for _ in range(3))
    got = oracle_mod.attention_fwd(Q, K, V, sm_scale=0.25, causal=True)
    assert np.array_equal(got[:, :, 0].view(np.uint16), V[:, :, 0].view(np.uint16))


def test_large_score_gap_saturates(oracle_mod):
    # scores 0 and 40: the second key's weight is 1 - e^-40, the first value's
    # share is below half an fp16 ulp, so the output is the second value row
    Q = np.array([[[[1.0, 0.0], [1.0, 0.0]]]], np.float16)
    K = np.array([[[[0.0, 5.0], [40.0, -3.0]]]], np.float16)
    V = np.array([[[[3.0, -7.0], [1.5, 0.25]]]], np.float16)
    got = oracle_mod.attention_fwd(Q, K, V, sm_scale=1.0, causal=False)
    assert np.array_equal(got[0, 0, 0], np.array([1.5, 0.25], np.float16))


# --------------------------------------------------------------------------
# Hand-derived cases
# --------------------------------------------------------------------------

def _hand_cases():
    with open(os.path.join(HERE, "golden", "attention_cases.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _hand_cases(), ids=lambda c: c["name"])
def test_hand_cases(oracle_mod, case):
    Q = np.array(case["Q"], np.float16)[None, None]
    K = np.array(case["K"], np.float16)[None, None]
    V = np.array(case["V"], np.float16)[None, None]
    sm_scale = math.log(2.0) if case["sm_scale"] == "ln2" else float(case["sm_scale"])
    got = oracle_mod.attention_fwd(Q, K, V, sm_scale=sm_scale, causal=bool(case["causal"]))[0, 0]
    assert np.array_equal(got.view(np.uint16), np.array(case["O_bits"], np.uint16))


# --------------------------------------------------------------------------
# Invariants
# --------------------------------------------------------------------------

def test_joint_key_value_permutation_leaves_output(oracle_mod):
    rng = np.random.default_rng(4)
    Q, K, V = (rng.standard_normal((2, 2, 33, 16)).astype(np.float16) for _ in range(3))
    perm = rng.permutation(33)
    a = oracle_mod.attention_fwd(Q, K, V, sm_scale=0.25, causal=False)
    b = oracle_mod.attention_fwd(Q, K[:, :, perm], V[:, :, perm], sm_scale=0.25, causal=False)
    # the fp64 sums run in another order: at most one fp16 ulp apart
    assert ulp_diff(a, b).max() <= 1


def test_factor_two_between_queries_and_scale(oracle_mod):
    rng = np.random.default_rng(5)
    Q, K, V = (rng.standard_normal((1, 3, 20, 8)).astype(np.float16) for _ in range(3))
    a = oracle_mod.attention_fwd((Q.astype(np.float32) * 2).astype(np.float16), K, V, sm_scale=0.125, causal=True)
    b = oracle_mod.attention_fwd(Q, K, V, sm_scale=0.25, causal=True)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


def test_row_selection_matches_full_result(oracle_mod):
    rng = np.random.default_rng(6)
    Q, K, V = (rng.standard_normal((2, 3, 10, 8)).astype(np.float16) for _ in range(3))
    full = oracle_mod.attention_fwd(Q, K, V, sm_scale=0.3, causal=True).reshape(-1, 8)
    rows = [59, 0, 17, 17, 31]
    part = oracle_mod.attention_fwd(Q, K, V, sm_scale=0.3, causal=True, rows=rows)
    assert np.array_equal(part.view(np.uint16), full.view(np.uint16)[rows])


# --------------------------------------------------------------------------
# Sensitivity: plausible mistakes must fail pin data
# --------------------------------------------------------------------------

def _restated(Q, K, V, sm_scale, causal, mistake=None):
    q, k, v = (x.astype(np.float64) for x in (Q, K, V))
    B, H, S, D = q.shape
    out = np.empty_like(q)
    for b in range(B):
        for h in range(H):
            s = (1.0 if mistake == "no_scale" else sm_scale) * q[b, h] @ k[b, h].T
            if causal:
                off = 0 if mistake != "causal_off_by_one" else -1
                s = np.where(np.arange(S)[None, :] <= np.arange(S)[:, None] + off, s, -np.inf)
            if mistake == "softmax_over_queries":
                p = np.exp(s - s.max(axis=0, keepdims=True))
                p = p / p.sum(axis=0, keepdims=True)
            else:
                m = 0.0 if mistake == "no_max" else s.max(axis=1, keepdims=True)
                p = np.exp(s - m)
                p = p / p.sum(axis=1, keepdims=True)
            vv = v[b, h][::-1] if mistake == "values_reversed" else v[b, h]
            out[b, h] = p @ vv
    with np.errstate(all="ignore"):
        return out.astype(np.float16)


@pytest.mark.parametrize("mistake", ["no_scale", "causal_off_by_one", "softmax_over_queries", "no_max",
                                     "values_reversed"])
def test_pins_catch_planted_mistakes(oracle_mod, mistake):
    rng = np.random.default_rng(7)
    S, D = 8, 4
    Q = rng.standard_normal((1, 1, S, D)).astype(np.float16)
    Q[0, 0, 3] = 30000.0    # a row with scores beyond exp's range: overflows without the max subtraction
    K = rng.standard_normal((1, 1, S, D)).astype(np.float16)
    V = rng.standard_normal((1, 1, S, D)).astype(np.float16)
    causal = mistake == "causal_off_by_one"
    truth = oracle_mod.attention_fwd(Q, K, V, sm_scale=0.5, causal=causal)
    assert ulp_diff(_restated(Q, K, V, 0.5, causal), truth).max() <= 1          # the harness is right
    bad = _restated(Q, K, V, 0.5, causal, mistake)
    assert (not np.isfinite(bad.astype(np.float64)).all()) or ulp_diff(bad, truth).max() > 1
