"""GPU unit test of the operand-tile layout: what TMA writes into shared memory.

The GEMM loads A boxes of 64 (K) x 128 (M) and B boxes of 64 (N) x 64 (K)
with the 128-byte swizzle, and its MMA descriptors read them assuming that
row r of a box starts at byte r * 128 and that its 16-byte piece j sits at
piece position j ^ (r % 8).  The nxmr.cn A100 article (sections 3.3 and 6.2)
describes what goes wrong when a shared-memory layout disagrees with the copy
engine's swizzle: rows shifted by 16 bytes.  gemm_f16_tma_box_image loads one
box exactly as the GEMM does and returns the raw shared-memory image, which
is checked here byte for byte against that formula, zero fill outside the
matrix included, for both operand box shapes and at ragged and negative
origins.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

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


def coded_matrix(rows, cols, seed):
    """Distinct finite binary16 patterns: element (r, c) is recognisable."""
    rng = np.random.default_rng(seed)
    codes = (np.arange(rows * cols, dtype=np.int64) * 7919 + int(rng.integers(0, 1 << 14))) % 0x7800 + 1
    return codes.astype(np.uint16).reshape(rows, cols)


def expected_image(X: np.ndarray, box_rows: int, x: int, y: int) -> np.ndarray:
    """The 128-byte-swizzled image of the box at (x, y), written out from the
    layout rule: element (y + r, x + c) goes to byte
    r * 128 + ((c // 8) ^ (r % 8)) * 16 + (c % 8) * 2; outside X it is 0."""
    rows, cols = X.shape
    img = np.zeros(box_rows * 64, dtype=np.uint16)
    for r in range(box_rows):
        for c in range(64):
            gr, gc = y + r, x + c
            v = X[gr, gc] if (0 <= gr < rows and 0 <= gc < cols) else 0
            img[r * 64 + ((c // 8) ^ (r % 8)) * 8 + (c % 8)] = v
    return img


CASES = [
    # (rows, cols, box_rows, x, y): A boxes (128 rows of 64 K values), B boxes (64 x 64)
    (512, 256, 128, 64, 128),      # interior A box
    (512, 256, 64, 128, 64),       # interior B box
    (1000, 1000, 128, 960, 896),   # ragged corner: 40 columns and 104 rows inside
    (300, 136, 64, 128, 256),      # 8 columns and 44 rows inside
    (200, 64, 128, -8, -5),        # negative origin: zero-filled top rows and first 8 columns
    (64, 64, 64, 64, 0),           # wholly outside: all zeros
    (37, 8, 16, 0, 30),            # a matrix narrower than the box
]


@pytest.mark.parametrize("rows,cols,box_rows,x,y", CASES)
def test_box_image_matches_the_swizzle_formula(g, rows, cols, box_rows, x, y):
    X = coded_matrix(rows, cols, seed=rows + cols)
    Xd = torch.from_numpy(X.view(np.float16)).to(DEV)
    img = g.tma_box_image(Xd, box_rows, x, y)
    assert g.check() == g.GEMM_OK
    got = img.cpu().numpy().view(np.uint16)
    want = expected_image(X, box_rows, x, y)
    if not np.array_equal(got, want):
        bad = np.flatnonzero(got != want)
        raise AssertionError(f"{len(bad)} of {want.size} elements misplaced; first at image element {bad[0]}: "
                             f"got {got[bad[0]]:#06x} want {want[bad[0]]:#06x}")


def test_formula_is_not_the_identity(g):
    # the swizzle really moves pieces: an unswizzled (plain row-major) reading
    # of the image differs from the box in every row but the multiples of 8
    X = coded_matrix(256, 128, seed=5)
    img = g.tma_box_image(torch.from_numpy(X.view(np.float16)).to(DEV), 64, 64, 0).cpu().numpy().view(np.uint16)
    plain = X[0:64, 64:128].reshape(-1)
    rows_equal = [np.array_equal(img[r * 64:(r + 1) * 64], plain[r * 64:(r + 1) * 64]) for r in range(64)]
    assert rows_equal == [r % 8 == 0 for r in range(64)]


def test_rejected_arguments_launch_nothing(g):
    X = torch.zeros((64, 64), dtype=torch.float16, device=DEV)
    for kwargs in ({"box_rows": 0, "x": 0, "y": 0}, {"box_rows": 257, "x": 0, "y": 0}):
        with pytest.raises(g.GemmError) as e:
            g.tma_box_image(X, **kwargs)
        assert e.value.status == g.GEMM_ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as e:
        g.tma_box_image(X, 16, 4, 0)   # x not on a 16-byte boundary
    assert e.value.status == g.GEMM_ERR_ALIGNMENT
    assert g.check() == g.GEMM_OK
