"""GPU parity of the attention forward against the CPU oracle.

Definition: the FlashAttention loop of the TileLang-MUSA lesson (7yue.com,
section 5): O = softmax(sm_scale Q K^T) V per (batch, head), keys j <= i when
causal.  Tolerance |gpu - ref| <= 6e-3 + 2e-3 |ref|, from the arithmetic: the
probabilities are rounded to fp16 for the P V product (relative error
<= 2^-11 per weight, so at most 2^-11 max|V| in the normalised sum, about
2.8e-3 for |V| <= 5.8, the largest N(0,1) draw in these tensors), the output
rounds once to fp16 (<= 2^-11 |O|), the 2^x unit and fp32 sums add far less;
the bound is doubled for margin.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from dense_fp16_gemm_05_gb300.inputs import ATTN_WORKLOADS, draw_attention, draw_attention_workload

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
ATOL, RTOL = 6e-3, 2e-3


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from dense_fp16_gemm_05_gb300 import build as gbuild
    gbuild.build()
    from dense_fp16_gemm_05_gb300 import gemm_f16
    gemm_f16.lib()
    return gemm_f16


def run(g, Q, K, V, causal, sm_scale=None):
    O = g.attention_fwd(Q.to(DEV), K.to(DEV), V.to(DEV), sm_scale=sm_scale, causal=causal)
    assert g.check() == g.GEMM_OK
    return O.cpu().numpy()


def assert_close(got, ref, what):
    got64, ref64 = got.astype(np.float64), ref.astype(np.float64)
    assert got.shape == ref.shape, what
    assert np.isfinite(got64).all(), f"{what}: non-finite output"
    err = np.abs(got64 - ref64)
    bad = err > ATOL + RTOL * np.abs(ref64)
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside tolerance, max err {err.max():.4g}"


@pytest.mark.parametrize("name,causal", [("attn_small_d64", False), ("attn_small_d64", True),
                                         ("attn_causal_ragged_d128", True), ("attn_causal_ragged_d128", False)])
def test_workloads_full(g, name, causal):
    w = ATTN_WORKLOADS[name]
    Q, K, V = draw_attention_workload(w)
    ref = oracle.attention_fwd(Q, K, V, sm_scale=w.sm_scale, causal=causal)
    assert_close(run(g, Q, K, V, causal, w.sm_scale), ref, f"{name} causal={causal}")


@pytest.mark.parametrize("name", ["attn_4096_d128", "attn_4096_d128_causal", "attn_4096_d64", "attn_4096_d64_causal"])
def test_4096_sampled_rows(g, name):
    w = ATTN_WORKLOADS[name]
    Q, K, V = draw_attention_workload(w)
    got = run(g, Q, K, V, w.causal, w.sm_scale).reshape(-1, w.dim)
    rng = np.random.default_rng(1)
    S = w.seq
    fixed = [0, 1, 127, 128, 2047, S - 1, S * w.heads * w.batch - 1, S * 5 + 3000]
    rows = sorted(set(fixed) | set(int(r) for r in rng.integers(0, got.shape[0], 16)))
    ref = oracle.attention_fwd(Q, K, V, sm_scale=w.sm_scale, causal=w.causal, rows=rows)
    assert_close(got[rows], ref, name)


@pytest.mark.parametrize("seq", [1, 2, 127, 128, 129, 255, 384])
@pytest.mark.parametrize("dim", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_edge_lengths(g, seq, dim, causal):
    Q, K, V = draw_attention(2, 2, seq, dim, seed=seq * 10 + dim + int(causal))
    sm = 1.0 / np.sqrt(dim)
    ref = oracle.attention_fwd(Q, K, V, sm_scale=sm, causal=causal)
    assert_close(run(g, Q, K, V, causal, sm), ref, f"seq {seq} dim {dim} causal {causal}")


@pytest.mark.parametrize("seq", [640, 1152])
@pytest.mark.parametrize("causal,queue", [(False, None), (True, None), (True, False)])
def test_many_items_per_cta(g, seq, causal, queue):
    # 3 x 40 heads: more work items than CTAs, so every CTA walks several;
    # with the causal mask an odd count of query-block pairs (3 and 5) leaves
    # a middle pair with no partner in its head (fixed shares), and the work
    # queue hands out 120 x 3 or 120 x 5 items
    Q, K, V = draw_attention(3, 40, seq, 64, seed=seq + int(causal))
    ref = oracle.attention_fwd(Q, K, V, sm_scale=0.125, causal=causal)
    O = g.attention_fwd(Q.to(DEV), K.to(DEV), V.to(DEV), sm_scale=0.125, causal=causal, queue=queue)
    assert g.check() == g.GEMM_OK
    assert_close(O.cpu().numpy(), ref, f"3x40 heads seq {seq} causal {causal} queue {queue}")


def _fixed_and_queued(g, shape, seed, qt):
    Q, K, V = (t.to(DEV) for t in draw_attention(*shape, seed=seed))
    fixed = g.attention_fwd(Q, K, V, causal=True, queue=False)
    queued = g.attention_fwd(Q, K, V, causal=True, queue=qt)
    return fixed, queued


@pytest.mark.parametrize("shape", [(3, 40, 1152, 64), (1, 24, 2048, 128), (4, 32, 4096, 128)])
def test_queue_gives_the_fixed_shares_bits_and_ends_zero(g, shape):
    # the queue changes which SM computes a pair of query blocks, not how
    qt = torch.zeros(2, dtype=torch.int32, device=DEV)
    fixed, queued = _fixed_and_queued(g, shape, 300 + shape[2], qt)
    assert g.check() == g.GEMM_OK
    assert torch.equal(fixed, queued), f"{shape}: queue and fixed shares differ"
    assert qt.cpu().tolist() == [0, 0]


def test_one_queue_for_back_to_back_launches(g):
    # three launches of different sizes share one queue on one stream with no
    # synchronisation between them; each leaves it zero for the next
    qt = torch.zeros(2, dtype=torch.int32, device=DEV)
    shapes = [(2, 8, 4096, 128), (3, 40, 640, 64), (1, 4, 129, 128)]
    inputs = [tuple(t.to(DEV) for t in draw_attention(*sh, seed=400 + i)) for i, sh in enumerate(shapes)]
    queued = [g.attention_fwd(Q, K, V, causal=True, queue=qt) for Q, K, V in inputs]
    fixed = [g.attention_fwd(Q, K, V, causal=True, queue=False) for Q, K, V in inputs]
    assert g.check() == g.GEMM_OK
    for sh, a, b in zip(shapes, queued, fixed):
        assert torch.equal(a, b), f"{sh}: queue and fixed shares differ"
    assert qt.cpu().tolist() == [0, 0]


def test_concurrent_streams_each_with_its_own_queue(g):
    # two causal launches in flight on two streams, each with the binding's
    # own fresh queue (made on its launch stream)
    shapes = [(2, 16, 2048, 128), (3, 20, 1536, 64)]
    inputs = [tuple(t.to(DEV) for t in draw_attention(*sh, seed=500 + i)) for i, sh in enumerate(shapes)]
    expect = [g.attention_fwd(Q, K, V, causal=True, queue=False) for Q, K, V in inputs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for _ in range(3):
        for st, (Q, K, V) in zip(streams, inputs):
            st.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(st):
                outs.append(g.attention_fwd(Q, K, V, causal=True))
    torch.cuda.synchronize()
    assert g.check() == g.GEMM_OK
    for i, o in enumerate(outs):
        assert torch.equal(o, expect[i % 2]), f"launch {i}"


@pytest.mark.parametrize("explicit_queue", [True, False])
def test_queue_inside_a_cuda_graph(g, explicit_queue):
    # captured once and replayed three times: an explicit queue is left zero
    # by every replay; the binding's own queue is zeroed by a captured fill
    Q, K, V = (t.to(DEV) for t in draw_attention(2, 24, 1536, 128, seed=77))
    expect = g.attention_fwd(Q, K, V, causal=True, queue=False)
    O = torch.empty_like(Q)
    qt = torch.zeros(2, dtype=torch.int32, device=DEV) if explicit_queue else None
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    cg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cg, stream=s):
        g.attention_fwd(Q, K, V, O=O, causal=True, queue=qt)
    for _ in range(3):
        O.fill_(float("nan"))
        cg.replay()
        torch.cuda.synchronize()
        assert g.check() == g.GEMM_OK
        assert torch.equal(O, expect)
    if explicit_queue:
        assert qt.cpu().tolist() == [0, 0]


def test_queue_arguments_rejected(g):
    Q, K, V = (t.to(DEV) for t in draw_attention(1, 2, 256, 64, seed=5))
    O = torch.empty_like(Q)
    L = g.lib()
    qt = torch.zeros(4, dtype=torch.int32, device=DEV)
    args = (Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), 1, 2, 256, 64, 0.125, 1)
    assert L.attention_fwd_f16_queue(*args, qt.data_ptr() + 2, None) == g.GEMM_ERR_ALIGNMENT
    assert L.attention_fwd_f16_queue(*args, O.data_ptr() + 64, None) == g.GEMM_ERR_INVALID_ARG   # inside O
    assert L.attention_fwd_f16_queue(*args, K.data_ptr(), None) == g.GEMM_ERR_INVALID_ARG        # inside K
    # not causal: the queue is not used, so not checked
    nc = args[:-1] + (0,)
    assert L.attention_fwd_f16_queue(*nc, qt.data_ptr() + 2, None) == g.GEMM_OK
    assert g.check() == g.GEMM_OK
    with pytest.raises(ValueError):
        g.attention_fwd(Q, K, V, causal=True, queue=torch.zeros(2, dtype=torch.int64, device=DEV))
    with pytest.raises(ValueError):
        g.attention_fwd(Q, K, V, causal=True, queue=torch.zeros(1, dtype=torch.int32, device=DEV))


def test_zero_queries_average_the_values(g):
    Q = torch.zeros((1, 4, 300, 128), dtype=torch.float16)
    _, K, V = draw_attention(1, 4, 300, 128, seed=77)
    got = run(g, Q, K, V, False).astype(np.float64)
    mean = V.double().mean(dim=2, keepdim=True).expand_as(V).numpy()
    assert np.abs(got - mean).max() <= ATOL


@pytest.mark.parametrize("queue", [None, False])
def test_causal_first_row_is_the_first_value_row(g, queue):
    # with the causal mask row 0 sees key 0 alone: weight 1, so O[.., 0, :]
    # is V[.., 0, :] exactly, for every head, at the bench's size
    w = ATTN_WORKLOADS["attn_4096_d128_causal"]
    Q, K, V = (t.to(DEV) for t in draw_attention_workload(w))
    O = g.attention_fwd(Q, K, V, sm_scale=w.sm_scale, causal=True, queue=queue)
    assert g.check() == g.GEMM_OK
    assert torch.equal(O[:, :, 0, :], V[:, :, 0, :])


@pytest.mark.parametrize("dim", [64, 128])
def test_causal_zero_queries_give_prefix_means(g, dim):
    # zero queries: equal scores, so row i averages V[0..i]
    B, H, S = 2, 3, 1000
    Q = torch.zeros((B, H, S, dim), dtype=torch.float16)
    _, K, V = draw_attention(B, H, S, dim, seed=90 + dim)
    got = run(g, Q, K, V, True).astype(np.float64)
    v = V.double().numpy()
    mean = np.cumsum(v, axis=2) / np.arange(1, S + 1).reshape(1, 1, S, 1)
    assert np.abs(got - mean).max() <= ATOL


def test_large_scores_do_not_overflow(g):
    # scores up to ~ 3e4: the running maximum keeps every exponent <= 8
    Q, K, V = draw_attention(1, 2, 256, 64, seed=78)
    Q = Q * 60.0
    ref = oracle.attention_fwd(Q.half(), K, V, sm_scale=0.125, causal=False)
    assert_close(run(g, Q.half(), K, V, False, 0.125), ref, "large scores")


def test_rejected_arguments(g):
    Q = torch.zeros((1, 1, 64, 96), dtype=torch.float16, device=DEV)
    with pytest.raises(g.GemmError) as e:
        g.attention_fwd(Q, Q.clone(), Q.clone())
    assert e.value.status == g.GEMM_ERR_INVALID_ARG
    Q = torch.zeros((1, 1, 64, 64), dtype=torch.float16, device=DEV)
    with pytest.raises(g.GemmError):
        g.attention_fwd(Q, Q.clone(), Q.clone(), O=Q)          # O overlaps Q
    E = torch.zeros((1, 1, 0, 64), dtype=torch.float16, device=DEV)
    g.attention_fwd(E, E, E)                                   # empty: no-op
    assert g.check() == g.GEMM_OK
