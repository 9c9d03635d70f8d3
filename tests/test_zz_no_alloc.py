"""GPU test of gemm_f16_ex_noalloc, the GEMM entry point that never allocates.

Some callers of a GEMM may not allocate device memory while they run: code
that reserved its whole memory budget up front (a serving process whose pool
already holds the GPU's memory, where a stream-ordered allocation from the
default pool can fail), plug-ins whose host framework forbids allocation in
their execute step, and latency-bound loops that must not go through the
allocator at all.  For them the K-slice partials of a split GEMM live in the
library's fixed 16 MiB device scratch instead of a per-call workspace.

Collected last (file name) so that it also runs after every other GPU test in
the same process; it passes alone as well.  Every call must give exactly the
bits of gemm_f16_ex with the same configuration (same kernels, same slice
order), also when several calls follow each other on one stream with no
synchronisation in between, so stale scratch contents from an earlier call
can never leak into a result.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from dense_fp16_gemm_05_gb300.inputs import draw

pytestmark = pytest.mark.gpu

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


def both(g, M, N, K, config, seed, relu=True):
    A, B = (x.to(DEV) for x in draw(M, N, K, "normal_scaled", seed))
    ref = g.gemm_f16(A, B, relu=relu, config=config)
    C = torch.full((M, N), 3.0, dtype=torch.float16, device=DEV)
    g.gemm_f16_noalloc(A, B, C, relu=relu, config=config)
    assert g.check() == g.GEMM_OK
    return A, B, ref.cpu().numpy(), C.cpu().numpy()


def test_two_consecutive_calls_match_the_allocating_entry_point(g):
    # 4 x 1024 x 1024 floats = 16 MiB: the scratch exactly; then a smaller
    # problem with more slices, which reads none of the first call's data
    for (M, N, K, cfg, seed) in [(1024, 1024, 4096, 2 | g.ksplit(4), 1), (512, 512, 8192, 3 | g.ksplit(8), 2)]:
        A, B, ref, got = both(g, M, N, K, cfg, seed)
        assert np.array_equal(got.view(np.uint16), ref.view(np.uint16)), (M, N, K, hex(cfg))
        rows = [0, M // 2, M - 1]
        want = oracle.gemm_f16(A.cpu(), B.cpu(), relu=True, rows=rows).astype(np.float64)
        assert np.all(np.abs(got[rows].astype(np.float64) - want) <= 2e-2 + 2e-3 * np.abs(want))


def test_repeated_call_same_problem_same_bits(g):
    cfg = 2 | g.GEMM_F16_KSPLIT_AUTO
    _, _, ref, first = both(g, 256, 512, 16384, cfg, 3, relu=False)
    _, _, _, second = both(g, 256, 512, 16384, cfg, 3, relu=False)
    assert np.array_equal(first.view(np.uint16), ref.view(np.uint16))
    assert np.array_equal(second.view(np.uint16), first.view(np.uint16))


def test_without_split_it_is_the_plain_call(g):
    _, _, ref, got = both(g, 384, 256, 2048, 2 | g.GEMM_F16_NO_KSPLIT, 4)
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))


def test_oversize_split_is_rejected_before_launch(g):
    # 8 x 1024 x 1024 floats = 32 MiB > 16 MiB
    A, B = (x.to(DEV) for x in draw(1024, 1024, 4096, "normal_scaled", 5))
    C = torch.full((1024, 1024), 3.0, dtype=torch.float16, device=DEV)
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16_noalloc(A, B, C, config=2 | g.ksplit(8))
    assert e.value.status == g.GEMM_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(C == 3.0)
    assert g.check() == g.GEMM_OK


def test_back_to_back_calls_without_sync(g):
    # three different split problems enqueued one after the other on one
    # stream: each GEMM's slices overwrite the scratch the previous call's
    # reduction read, which stream order (and the kernels' dependency waits)
    # must keep apart
    k = g.ksplit
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    # a tail split on the 128 x 128 configuration: one full wave of tiles, then
    # a remainder of about a third of the slots, cut into K slices
    m_tail = 128 * ((sms + sms // 3) // 8 + 1)
    tiles = (m_tail // 128) * 8
    rest = tiles - sms
    assert 2 <= sms // rest and rest * min(sms // rest, 5) * 128 * 128 * 4 <= 16 << 20
    problems = [(1024, 1024, 4096, 2 | k(4), 11, True),
                (m_tail, 1024, 3000, 2 | g.GEMM_F16_KSPLIT_TAIL, 12, False),
                (512, 768, 8192, 3 | k(8), 13, True)]
    ins, refs = [], []
    for (M, N, K, cfg, seed, relu) in problems:
        A, B = (x.to(DEV) for x in draw(M, N, K, "normal_scaled", seed))
        ins.append((A, B, torch.full((M, N), 7.0, dtype=torch.float16, device=DEV)))
        refs.append(g.gemm_f16(A, B, relu=relu, config=cfg))
    assert g.check() == g.GEMM_OK
    for (A, B, C), (M, N, K, cfg, seed, relu) in zip(ins, problems):
        g.gemm_f16_noalloc(A, B, C, relu=relu, config=cfg)
    assert g.check() == g.GEMM_OK
    for (A, B, C), ref, prob in zip(ins, refs, problems):
        assert torch.equal(C.view(torch.int16), ref.view(torch.int16)), prob


def test_rule_chosen_split_and_automatic_choice(g):
    # 1024 x 1024 x 16384 on the 256 x 256 pair configuration with the slice
    # rule: 16 tiles x 4 slices of 256 x 256 fp32 partials fill the scratch
    # exactly; configuration 0 (which never takes a workspace split) gives
    # the bits of gemm_f16
    A, B = (x.to(DEV) for x in draw(1024, 1024, 16384, "normal_scaled", 14))
    for cfg in (3 | g.GEMM_F16_KSPLIT_AUTO, 0):
        ref = g.gemm_f16(A, B, relu=True, config=cfg)
        C = torch.empty_like(ref)
        g.gemm_f16_noalloc(A, B, C, relu=True, config=cfg)
        assert g.check() == g.GEMM_OK
        assert torch.equal(C.view(torch.int16), ref.view(torch.int16)), hex(cfg)
