"""Host-only checks of the C ABI (no GPU needed, no kernel launched).

The library must load on a machine without a GPU driver, export every
function that include/gemm_f16.h declares, and reject bad arguments before
touching the GPU.
"""
from __future__ import annotations

import ctypes
import re

import pytest

from dense_fp16_gemm_05_gb300 import build as gbuild


@pytest.fixture(scope="module")
def g():
    gbuild.build()
    from dense_fp16_gemm_05_gb300 import gemm_f16
    gemm_f16.lib()
    return gemm_f16


def test_library_exports_every_declared_function(g):
    names = g.header_functions()
    assert "gemm_f16" in names and "gemm_f16_check" in names
    raw = ctypes.CDLL(gbuild.LIB)
    missing = [n for n in names if not hasattr(raw, n)]
    assert not missing, missing


def test_header_declarations_are_extern_c_and_plain_types():
    with open(gbuild.os.path.join(gbuild.INCLUDE, "gemm_f16.h")) as f:
        text = f.read()
    assert 'extern "C"' in text
    assert "torch" not in re.sub(r"/\*.*?\*/", "", text, flags=re.S)


def test_version_matches_header(g):
    with open(g.HEADER) as f:
        m = re.search(r"#define GEMM_F16_VERSION (\d+)", f.read())
    assert g.version() == int(m.group(1))


def test_strerror_covers_all_codes(g):
    for code in (0, -1, -2, -3, -4, -5, -6):
        s = g.strerror(code)
        assert s and s != "unknown status"
    assert g.strerror(-99) == "unknown status"


def test_configs_are_named(g):
    n = g.num_configs()
    assert n >= 1
    assert g.config_name(0) == "auto"
    for i in range(1, n + 1):
        assert g.config_name(i)
    assert g.config_name(n + 1) is None and g.config_name(-1) is None


@pytest.mark.parametrize("M,N,K", [(-1, 8, 8), (8, -1, 8), (8, 8, -1), (2**31, 8, 8), (8, 2**31, 8),
                                   (8, 8, 2**31)])
def test_bad_sizes_rejected_before_any_cuda_call(g, M, N, K):
    assert g.gemm_f16_raw(0, 0, 0, M, N, K, 1) == g.GEMM_ERR_INVALID_ARG


def test_cluster_k_configuration_is_named_without_cuda(g):
    ck = [c for c in range(1, g.num_configs() + 1) if g.config_cluster_k(c)]
    assert len(ck) == 1 and "_ck" in g.config_name(ck[0])
    assert g.config_layouts(ck[0]) == 0x1
    assert ck[0] not in g.workspace_split_configs()
    assert not g.config_cluster_k(0)
    with pytest.raises(g.GemmError):
        g.config_cluster_k(g.num_configs() + 1)


def test_bad_relu_and_config_rejected(g):
    assert g.gemm_f16_raw(0, 0, 0, 8, 8, 8, 2) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_f16_raw(0, 0, 0, 8, 8, 8, -1) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_f16_raw(0, 0, 0, 8, 8, 8, 1, config=g.num_configs() + 1) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_f16_raw(0, 0, 0, 8, 8, 8, 1, config=-1) == g.GEMM_ERR_INVALID_ARG


def test_empty_problem_is_a_no_op(g):
    # M == 0 or N == 0 touches nothing, so even NULL pointers are fine
    assert g.gemm_f16_raw(0, 0, 0, 0, 8, 8, 1) == g.GEMM_OK
    assert g.gemm_f16_raw(0, 0, 0, 8, 0, 8, 1) == g.GEMM_OK


def test_no_gpu_gives_a_status_not_a_crash(g):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = g.gemm_f16_raw(16, 16, 16, 8, 8, 8, 1)
    assert st in (g.GEMM_ERR_CUDA, g.GEMM_ERR_UNSUPPORTED_DEVICE)


def test_binding_fails_loudly_without_library(monkeypatch):
    from dense_fp16_gemm_05_gb300 import gemm_f16 as mod
    monkeypatch.setattr(mod, "_lib", None)
    monkeypatch.setattr(mod._build, "LIB", "/nonexistent/libgemm_f16.so")
    with pytest.raises(mod.LibraryNotBuilt):
        mod.lib()


def test_selftest_timeout_rejects_bad_budgets_before_any_cuda_call(g):
    L = g.lib()
    # K == 0 or out-of-range budgets are refused without touching the GPU
    assert L.gemm_f16_selftest_timeout(None, None, None, 64, 64, 0, 0, 1 << 20, None) == g.GEMM_ERR_INVALID_ARG
    assert L.gemm_f16_selftest_timeout(None, None, None, 64, 64, 64, 0, 100, None) == g.GEMM_ERR_INVALID_ARG
    assert L.gemm_f16_selftest_timeout(None, None, None, 64, 64, 64, 0, 1 << 40, None) == g.GEMM_ERR_INVALID_ARG


def test_config_flag_constants_match_header(g):
    with open(g.HEADER) as f:
        text = f.read()
    assert int(re.search(r"#define GEMM_F16_CONFIG_ID_MASK (0x[0-9A-Fa-f]+)", text).group(1), 16) == \
        g.GEMM_F16_CONFIG_ID_MASK
    assert int(re.search(r"#define GEMM_F16_NO_SPLIT (0x[0-9A-Fa-f]+)", text).group(1), 16) == g.GEMM_F16_NO_SPLIT
    assert int(re.search(r"#define GEMM_F16_NO_KSPLIT (0x[0-9A-Fa-f]+)", text).group(1), 16) == g.GEMM_F16_NO_KSPLIT
    assert int(re.search(r"#define GEMM_F16_KSPLIT_AUTO (0x[0-9A-Fa-f]+)", text).group(1), 16) == \
        g.GEMM_F16_KSPLIT_AUTO
    assert int(re.search(r"#define GEMM_F16_KSPLIT_TAIL (0x[0-9A-Fa-f]+)", text).group(1), 16) == \
        g.GEMM_F16_KSPLIT_TAIL
    assert int(re.search(r"#define GEMM_F16_KSPLIT_SHIFT (\d+)", text).group(1)) == g.GEMM_F16_KSPLIT_SHIFT
    assert int(re.search(r"#define GEMM_F16_KSPLIT_MASK (0x[0-9A-Fa-f]+)", text).group(1), 16) == \
        g.GEMM_F16_KSPLIT_MASK
    assert g.ksplit(16) & ~g.GEMM_F16_KSPLIT_MASK == 0 and g.ksplit(2) >> g.GEMM_F16_KSPLIT_SHIFT == 2


def test_config_flags_parsed_before_cuda(g):
    # a known id with the no-split flag names the same configuration; an unknown
    # flag bit or id is rejected without touching the GPU
    for cfg in range(0, g.num_configs() + 1):
        assert g.config_name(cfg | g.GEMM_F16_NO_SPLIT) == g.config_name(cfg)
        assert g.config_layouts(cfg | g.GEMM_F16_NO_SPLIT) == g.config_layouts(cfg)
    assert g.config_name(1 | 0x20000) is None
    assert g.config_name(1 | 0x40000) is None
    assert g.config_name(g.num_configs() + 1) is None
    assert g.config_layouts(1 | 0x40000) == g.GEMM_ERR_INVALID_ARG
    st = g.lib().gemm_f16_ex(0, 0, 0, 64, 64, 64, 1, 1 | 0x40000, None)
    assert st == g.GEMM_ERR_INVALID_ARG


def test_ksplit_flags_parsed_before_cuda(g):
    # K-split counts 2..16 and the never-split flag name the same configuration;
    # a count of 1 or above 16, or both flags together, are rejected without a GPU
    for cfg in range(0, g.num_configs() + 1):
        for n in range(2, 17):
            assert g.config_name(cfg | g.ksplit(n)) == g.config_name(cfg)
        assert g.config_name(cfg | g.GEMM_F16_NO_KSPLIT) == g.config_name(cfg)
        assert g.config_name(cfg | g.GEMM_F16_KSPLIT_AUTO) == g.config_name(cfg)
        assert g.config_name(cfg | g.GEMM_F16_KSPLIT_TAIL) == g.config_name(cfg)
        assert g.config_name(cfg | g.GEMM_F16_NO_SPLIT | g.ksplit(4)) == g.config_name(cfg)
    for bad in (g.ksplit(1), g.ksplit(17), g.ksplit(31), g.GEMM_F16_NO_KSPLIT | g.ksplit(2),
                g.GEMM_F16_KSPLIT_AUTO | g.ksplit(2), g.GEMM_F16_KSPLIT_AUTO | g.GEMM_F16_NO_KSPLIT,
                g.GEMM_F16_KSPLIT_TAIL | g.ksplit(4), g.GEMM_F16_KSPLIT_TAIL | g.GEMM_F16_KSPLIT_AUTO,
                g.GEMM_F16_KSPLIT_TAIL | g.GEMM_F16_NO_KSPLIT):
        assert g.config_name(1 | bad) is None
        assert g.config_layouts(1 | bad) == g.GEMM_ERR_INVALID_ARG
    assert g.config_label(3 | g.ksplit(4)) == g.config_name(3) + "+ksplit4"


def _tuned_table():
    import os
    from dense_fp16_gemm_05_gb300 import build as gbuild
    path = os.path.join(gbuild.CSRC, "gemm_f16_tuned.inc")
    with open(path) as f:
        text = f.read()
    cands = [int(x, 16) for x in re.search(r"kTunedCandidates\[[^\]]*\] = \{([^}]*)\}", text).group(1).split(",")]
    rows = []
    for m in re.finditer(r"\{(\d+), (\d+), (\d+), \{([^}]*)\}\}", text):
        vals = [float(x.strip().rstrip("f")) for x in m.group(4).split(",")]
        rows.append((int(m.group(1)), int(m.group(2)), int(m.group(3)), vals))
    n_rows = int(re.search(r"#define GEMM_F16_TUNED_ROWS (\d+)", text).group(1))
    n_cands = int(re.search(r"#define GEMM_F16_TUNED_CANDIDATES (\d+)", text).group(1))
    return cands, rows, n_rows, n_cands


def test_tuned_table_is_well_formed(g):
    cands, rows, n_rows, n_cands = _tuned_table()
    assert len(cands) == n_cands and len(rows) == n_rows > 0
    for c in cands:
        assert 1 <= (c & g.GEMM_F16_CONFIG_ID_MASK) <= g.num_configs()
        assert (c & ~(g.GEMM_F16_CONFIG_ID_MASK | g.GEMM_F16_NO_SPLIT | g.GEMM_F16_KSPLIT_AUTO
                      | g.GEMM_F16_KSPLIT_TAIL | g.GEMM_F16_KSPLIT_MASK | g.GEMM_F16_NO_KSPLIT)) == 0
    shapes = [r[:3] for r in rows]
    assert len(set(shapes)) == len(shapes)
    for M, N, K, vals in rows:
        assert M > 0 and N > 0 and K > 0 and len(vals) == n_cands
        assert all(v > 0 for v in vals)


def test_fp8_arguments_rejected_before_cuda(g):
    L = g.lib()
    assert L.gemm_fp8_block_scaled(None, None, None, None, None, -1, 64, 64, 1, None) == g.GEMM_ERR_INVALID_ARG
    assert L.gemm_fp8_block_scaled(None, None, None, None, None, 64, 64, 64, 2, None) == g.GEMM_ERR_INVALID_ARG
    assert L.gemm_fp8_block_scaled(None, None, None, None, None, 0, 64, 64, 1, None) == g.GEMM_OK   # empty: no-op


def test_attention_arguments_rejected_before_cuda(g):
    L = g.lib()
    assert L.attention_fwd_f16(None, None, None, None, 1, 1, 64, 96, 0.1, 0, None) == g.GEMM_ERR_INVALID_ARG
    assert L.attention_fwd_f16(None, None, None, None, -1, 1, 64, 64, 0.1, 0, None) == g.GEMM_ERR_INVALID_ARG
    assert L.attention_fwd_f16(None, None, None, None, 1, 1, 64, 64, 0.1, 2, None) == g.GEMM_ERR_INVALID_ARG
    assert L.attention_fwd_f16(None, None, None, None, 1, 1, 64, 64, float("inf"), 0, None) == g.GEMM_ERR_INVALID_ARG
    assert L.attention_fwd_f16(None, None, None, None, 0, 1, 64, 64, 0.1, 0, None) == g.GEMM_OK
    Lq = L.attention_fwd_f16_queue
    assert Lq(None, None, None, None, 1, 1, 64, 96, 0.1, 1, None, None) == g.GEMM_ERR_INVALID_ARG
    assert Lq(None, None, None, None, 1, 1, 64, 64, 0.1, 2, None, None) == g.GEMM_ERR_INVALID_ARG
    assert Lq(None, None, None, None, 0, 1, 64, 64, 0.1, 1, None, None) == g.GEMM_OK
