"""Seeded random problems through the planner's own choices, every element
against the oracle: shapes from one element to a few thousand on each side,
every operand type, ragged and padded strides (TMA-legal and not), both
epilogues, random alpha; and the block-scaled types with random shapes.
Each case prints its plan, so a failure names the kernel and schedule."""

from __future__ import annotations

import numpy as np
import pytest

import seeded_inputs as si
from gemm_harness import check_full, check_mx

pytestmark = pytest.mark.gpu

DENSE = ["bf16", "fp16", "tf32", "e4m3", "e5m2"]
SCALED = ["e4m3", "e5m2", "e2m1", "nvf4"]


@pytest.fixture(scope="module", autouse=True)
def _library():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_gemm_epilogue_gb300 as tg

    tg.build()
    tg.load()


def _dim(rng) -> int:
    """Mostly small-to-mid sizes, with tile-edge values and a few large ones."""
    r = rng.random()
    if r < 0.15:
        return int(rng.integers(1, 9))
    if r < 0.35:
        return int(rng.choice([63, 64, 65, 127, 128, 129, 255, 256, 257, 511, 512, 513]))
    if r < 0.9:
        return int(rng.integers(9, 1500))
    return int(rng.integers(1500, 3000))


def _ld(rng, K: int, dtype: str) -> int:
    """A row stride >= K: mostly a 16-byte multiple (the TMA paths), else
    any padding (the plain-load producer)."""
    if rng.random() < 0.7:
        per16 = int(16 // si.element_bytes(dtype))
        return -(-K // per16) * per16 + per16 * int(rng.integers(0, 3))
    return K + int(rng.integers(0, 20))


def _dense_cases(n=48, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for c in range(n):
        dtype = DENSE[c % len(DENSE)]
        M, N, K = _dim(rng), _dim(rng), _dim(rng)
        if rng.random() < 0.15:        # many pair tiles, short K: tickets, two-pair clusters
            M, N, K = int(rng.integers(3000, 6000)), int(rng.integers(3000, 6000)), \
                int(rng.integers(16, 200))
        while M * N * K > 2.5e9:       # keep each oracle call to a second or two
            K = max(1, K // 2)
        lda, ldb, ldc = _ld(rng, K, dtype), _ld(rng, K, dtype), M + int(rng.choice([0, 1, 4]))
        alpha = float(rng.choice([1.0, -0.5, 1.75, 0.0625]))
        dist = "normal" if rng.random() < 0.5 else "uniform"
        out.append(si.Workload(f"fz{c}_{dtype}", M, N, K, dtype, alpha, bool(rng.random() < 0.6),
                               5000 + c, dist, lda=lda, ldb=ldb, ldc=ldc))
    # A few problems large enough for the many-wave CTA-pair schedules:
    # tickets (>= 6 waves, longer K loops) and two-pair clusters (short K).
    for c, (lo, hi, klo, khi) in enumerate([(5700, 6300, 2100, 2500), (5700, 6300, 2100, 2500),
                                            (4800, 5600, 600, 1900), (4800, 5600, 600, 1900)]):
        dtype = ("bf16", "fp16")[c % 2]
        M, N = int(rng.integers(lo, hi)), int(rng.integers(lo, hi))
        K = int(rng.integers(klo, khi))
        out.append(si.Workload(f"fzbig{c}_{dtype}", M, N, K, dtype, 1.0, True, 5900 + c, "normal",
                               lda=-(-K // 8) * 8 + 8 * (c & 1), ldb=-(-K // 8) * 8, ldc=M + 2))
    return out


def _scaled_cases(n=20, seed=77):
    rng = np.random.default_rng(seed)
    out = []
    for c in range(n):
        dtype = SCALED[c % len(SCALED)]
        M, N, K = _dim(rng), _dim(rng), _dim(rng)
        while M * N * K > 1.5e9:
            K = max(2, K // 2)
        if dtype in ("e2m1", "nvf4"):
            K += K & 1
        pad = int(rng.choice([0, 0, 2, 16, 32]))   # even: packed FP4 rows stay whole bytes
        lda, ldb = K + pad, K + int(rng.choice([0, 32]))
        out.append(si.Workload(f"fzs{c}_{dtype}", M, N, K, dtype, float(rng.choice([1.0, -1.25])),
                               bool(rng.random() < 0.6), 6000 + c, "normal", lda=lda, ldb=ldb,
                               ldc=M + int(rng.choice([0, 3])), block_scaled=True))
    return out


@pytest.mark.parametrize("w", _dense_cases(), ids=lambda w: f"{w.name}_{w.M}x{w.N}x{w.K}")
def test_random_dense_problem(w):
    import dense_gemm_epilogue_gb300 as tg

    lda, ldb, ldc = w.strides
    print(tg.tg_plan_describe(w.M, w.N, w.K, w.dtype, lda, ldb, ldc))
    check_full(w, repeats=2)


@pytest.mark.parametrize("w", _scaled_cases(), ids=lambda w: f"{w.name}_{w.M}x{w.N}x{w.K}")
def test_random_block_scaled_problem(w):
    check_mx(w, repeats=2)
