"""Failure detection on the GPU without a fault: a bounded wait that runs out.

gemm_f16_selftest_timeout launches the real kernel with its TMA producer
switched off and a short wait budget, so the MMA thread's first wait for
operand data can never be satisfied (a flag nothing sets).  The kernel must
record the wait site, leave every loop, free its tensor memory and exit
without touching C; gemm_f16_check must then report GEMM_ERR_TIMEOUT, and the
context must stay usable for a normal call right after.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from dense_fp16_gemm_05_gb300.inputs import draw

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
SITE_MMA_FULL = 3
SITE_EPILOGUE_TMEM_FULL = 4
SITE_CLUSTER_PARTIAL = 8


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from dense_fp16_gemm_05_gb300 import build as gbuild
    gbuild.build()
    from dense_fp16_gemm_05_gb300 import gemm_f16
    gemm_f16.lib()
    return gemm_f16


@pytest.mark.parametrize("config", [1, 3, 5, 6])
def test_wait_runs_out_and_context_survives(g, config):
    M, N, K = 512, 512, 256
    A, B = draw(M, N, K, "normal", seed=31)
    Ad, Bd = A.to(DEV), B.to(DEV)
    C = torch.full((M, N), 5.0, dtype=torch.float16, device=DEV)
    assert g.check() == g.GEMM_OK
    st = g.selftest_timeout(Ad, Bd, C, config=config, timeout_cycles=1 << 24)   # ~10 ms of SM clocks
    assert st == g.GEMM_OK
    assert g.check() == g.GEMM_ERR_TIMEOUT
    site = g.last_timeout_record() & 0xFF
    assert site in (SITE_MMA_FULL, SITE_EPILOGUE_TMEM_FULL, SITE_CLUSTER_PARTIAL), hex(g.last_timeout_record())
    # the aborted kernel stored nothing
    assert torch.all(C == 5.0)
    # the status word was cleared and the context still computes correctly
    assert g.check() == g.GEMM_OK
    g.gemm_f16(Ad, Bd, C, relu=True, config=config)
    assert g.check() == g.GEMM_OK
    got = C.cpu().numpy().astype(np.float64)
    ref = oracle.gemm_f16(A, B, relu=True).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2e-2 + 2e-3 * np.abs(ref))


def test_launch_geometry(g):
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    for config in range(1, g.num_configs() + 1):
        for (M, N, K) in [(8192, 8192, 8192), (1000, 1000, 1000), (64, 64, 64), (16384, 512, 64)]:
            info = g.launch_info(M, N, K, config)
            assert info["grid_ctas"] % info["cluster_size"] == 0
            assert info["tiles"] >= 1
            if g.config_cluster_k(config):
                # one cluster per tile
                assert info["grid_ctas"] == info["tiles"] * info["cluster_size"]
            else:
                assert 0 < info["grid_ctas"] <= sms   # persistent grid
    assert g.launch_info(8192, 8192, 8192, 3)["cluster_size"] == 2
    assert g.launch_info(8192, 8192, 8192, 1)["cluster_size"] == 1
