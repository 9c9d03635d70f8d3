"""GPU test: GEMMs that consume each other's results on one stream, with no
host synchronisation between them.

Every GEMM kernel (and the K-slice reduction) is launched as a programmatic
dependent of the kernel before it on the stream: its set-up may overlap the
end of that kernel, and it waits for that kernel's results before touching
memory.  A chain in which each GEMM reads the previous output checks that
the wait is in place for every kernel kind: a read of a stale or half-written
operand changes the result.

The chain is exact: C_1 = R(A @ B) on small integers (every partial sum
exact), then C_{i+1} = R(C_i @ P_i) with permutation matrices P_i, which only
move entries (C_i >= 0, so R changes nothing).  The expected result is the
oracle's C_1 with its columns permuted, compared bit for bit.
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


def chain_configs(g):
    k = g.ksplit
    return [0, 2, 3 | k(4), 5, 1 | k(3), 4, 5 | k(2), 6 | k(4), 2 | k(2), 6, 0, 5, 3, 1 | k(4), 6 | k(2)]


@pytest.mark.parametrize("graph", [False, True])
def test_dependent_chain_without_host_sync(g, graph):
    M, N, K = 384, 512, 128
    A, B = draw(M, N, K, "integer", seed=71)            # |partial sums| <= 16 * 128 = 2048: exact
    C1_ref = oracle.gemm_f16(A, B, relu=True)
    rng = np.random.default_rng(72)
    cfgs = chain_configs(g)
    perms = [rng.permutation(N) for _ in cfgs]
    P = []
    for perm in perms:
        m = np.zeros((N, N), dtype=np.float16)
        m[perm, np.arange(N)] = 1.0                     # (C @ m)[:, j] = C[:, perm[j]]
        P.append(torch.from_numpy(m).to(DEV))
    Ad, Bd = A.to(DEV), B.to(DEV)
    outs = [torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV) for _ in range(len(cfgs) + 1)]

    def run_chain():
        g.gemm_f16(Ad, Bd, C=outs[0], relu=True)
        for i, cfg in enumerate(cfgs):
            g.gemm_f16(outs[i], P[i], C=outs[i + 1], relu=True, config=cfg)

    if graph:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            run_chain()                                   # first calls outside the capture
        torch.cuda.synchronize()
        for o in outs:
            o.fill_(float("nan"))
        torch.cuda.synchronize()
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=s):
            run_chain()
        for o in outs:
            o.fill_(float("nan"))
        cg.replay()
    else:
        run_chain()
    assert g.check() == g.GEMM_OK
    expect = C1_ref.copy()
    got0 = outs[0].cpu().numpy()
    assert np.array_equal(got0.view(np.uint16), expect.view(np.uint16))
    for i, perm in enumerate(perms):
        expect = expect[:, perm]
        got = outs[i + 1].cpu().numpy()
        assert np.array_equal(got.view(np.uint16), expect.view(np.uint16)), f"step {i + 1} config {cfgs[i]:#x}"


def test_mixed_kernels_chain_matches_synchronised_run(g):
    # GEMM -> K-split GEMM -> cluster K-split GEMM -> ReLU gradient -> attention -> (torch cast) ->
    # FP8 GEMM -> GEMM, each reading the previous result.  Every kernel is
    # deterministic, so the chain run back to back must give the same bits as
    # the same chain with a device synchronisation after every call.
    from dense_fp16_gemm_05_gb300.inputs import draw_attention, draw_fp8_block_scaled
    n = 512
    A, B = draw(n, n, n, "normal_scaled", seed=81)
    B2 = draw(n, n, n, "normal_scaled", seed=82)[1]
    G = draw(n, n, n, "normal", seed=83)[0]
    _, Kt, Vt = draw_attention(1, 2, 1024, 128, seed=84)
    _, SA, W8, SW = draw_fp8_block_scaled(n, n, n, "normal", seed=85)
    Ad, Bd, B2d, Gd = (t.to(DEV) for t in (A, B, B2, G))
    Kd, Vd, SAd, W8d, SWd = (t.to(DEV) for t in (Kt, Vt, SA, W8, SW))

    def chain(sync):
        out = []
        def step(t):
            out.append(t)
            if sync:
                torch.cuda.synchronize()
            return t
        c1 = step(g.gemm_f16(Ad, Bd, relu=True, config=5))
        c2 = step(g.gemm_f16(c1, B2d, relu=False, config=2 | g.ksplit(4)))
        c2 = step(g.gemm_f16(c2, Bd, relu=False, config=6 | g.ksplit(4)))   # cluster K split
        dz = step(g.relu_backward(Gd, c2))
        o = step(g.attention_fwd(dz.view(1, 2, 1024, 128), Kd, Vd))
        a8 = o.view(n, n).to(torch.float8_e4m3fn)
        c3 = step(g.gemm_fp8_block_scaled(a8, SAd, W8d, SWd))
        step(g.gemm_f16(c3, Bd, relu=True, config=0))
        torch.cuda.synchronize()
        return [t.cpu() for t in out]

    free = chain(False)
    synced = chain(True)
    assert g.check() == g.GEMM_OK
    for i, (x, y) in enumerate(zip(free, synced)):
        assert not torch.isnan(y.float()).any(), f"step {i}: NaN"
        assert torch.equal(x.view(torch.int16), y.view(torch.int16)), f"step {i} differs from the synchronised run"
