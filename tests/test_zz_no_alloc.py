"""GPU test of gemm_f16_ex_noalloc, the entry point whose K-slice partials
live in the library's fixed 16 MiB device scratch instead of an allocation.

Collected last (file name) so that it also runs after every other GPU test in
the same process; it passes alone as well.  Two consecutive calls on
different problems must each give exactly the bits of gemm_f16_ex with the
same configuration (same kernels, same slice order), so stale scratch
contents from an earlier call can never leak into a result.
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
