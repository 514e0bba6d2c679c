"""8-bit float operands (E4M3 / E5M2, tcgen05.mma kind::f8f6f4) against the
oracle, element by element, through the C ABI.

The same coverage as the 16-bit kinds on a smaller scale: ragged edges,
every single-CTA tile configuration with both producers, CTA-pair tiles,
multicast clusters, split-K tails, swapped roles, batched calls with narrow
outputs, NaN and infinity codes, and the 8192^3 workload in full.
"""

from __future__ import annotations

import numpy as np
import pytest

import seeded_inputs as si
from gemm_harness import check_batched, check_full, logical, run_tg

pytestmark = pytest.mark.gpu
FP8 = ["e4m3", "e5m2"]


@pytest.fixture(scope="module", autouse=True)
def _library():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_gemm_epilogue_gb300 as tg

    tg.build()
    tg.load()


@pytest.mark.parametrize("dtype", FP8)
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (65, 97, 73), (129, 65, 33), (257, 255, 129),
                                   (17, 300, 70), (300, 520, 1040), (130, 140, 128)])
def test_fp8_edge_sweep(dtype, M, N, K):
    """Planner's choice; K = 73, 33, 129, 70 give TMA-illegal strides (plain
    loads), K = 1040 a ragged last K block on TMA."""
    w = si.Workload(f"f8edge_{dtype}", M, N, K, dtype, 1.5, True, 300 + M + 3 * N + K, "normal")
    check_full(w, repeats=2)


@pytest.mark.parametrize("dtype", FP8)
@pytest.mark.parametrize("block_n", [64, 128, 256])
@pytest.mark.parametrize("producer", [1, 2])
def test_fp8_every_config(dtype, block_n, producer):
    w = si.Workload("f8cfg", 300, 520, 400, dtype, -0.75, True, 61, "normal", lda=416, ldb=432,
                    ldc=304)
    check_full(w, opts={"block_n": block_n, "producer": producer, "cta_pair": 1})


@pytest.mark.parametrize("dtype", FP8)
@pytest.mark.parametrize("block_n", [128, 256])
@pytest.mark.parametrize("M,N,K", [(300, 520, 208), (513, 1000, 1040), (1, 17, 16),
                                   (600, 1100, 2048)])
def test_fp8_cta_pair(dtype, block_n, M, N, K):
    w = si.Workload("f8pair", M, N, K, dtype, 0.5, True, 71 + M + N, "normal", ldc=M + 3)
    check_full(w, opts={"cta_pair": 2, "block_n": block_n})


@pytest.mark.parametrize("dtype", FP8)
def test_fp8_multicast_and_swap(dtype):
    w = si.Workload("f8mc", 600, 1100, 1040, dtype, 1.25, True, 81, "normal", ldc=607)
    check_full(w, opts={"cta_pair": 2, "multicast": 2, "swap_ab": 1}, repeats=2)
    ws = si.Workload("f8swap", 64, 1000, 512, dtype, 1.0, False, 82, "normal")
    check_full(ws, opts={"swap_ab": 2})
    check_full(ws)


@pytest.mark.parametrize("dtype", FP8)
def test_fp8_split_k_tail(dtype):
    """Four pair tiles on all pairs: the planner cuts each into K segments."""
    import dense_gemm_epilogue_gb300 as tg

    w = si.Workload("f8split", 500, 500, 8192, dtype, 1.0, True, 83, "normal")
    lda, ldb, ldc = w.strides
    plan = tg.tg_plan(w.M, w.N, w.K, None, lda, None, ldb, None, ldc, dtype, {"cta_pair": 2})
    assert plan["block_k"] == 128 and plan["split_segs"] > 1
    check_full(w, opts={"cta_pair": 2}, repeats=3)


@pytest.mark.parametrize("dtype", FP8)
def test_fp8_batched_narrow_outputs(dtype):
    w = si.Workload("f8batch", 400, 700, 1024, dtype, 1.0, True, 84, "normal")
    for out in ("f32", "bf16", "fp16"):
        check_batched(w, 3, out)
    check_batched(w, 2, "bf16", share_b=True)


def test_fp8_nan_and_infinity_codes():
    """E4M3 S.1111.111 and E5M2 exponent-31 codes are NaN; E5M2 infinities
    give infinite sums (and NaN when met by a zero or an opposite infinity)."""
    for dtype in FP8:
        w = si.Workload("f8nan", 130, 70, 40, dtype, 1.0, True, 85, "normal")
        A, B = si.make_operands(w)
        A[5, 3] = np.uint8(0x7F)
        out = logical(run_tg(w, A, B), w)
        assert np.all(np.isnan(out[5, :]))
        assert not np.any(np.isnan(np.delete(out, 5, axis=0)))
    w = si.Workload("f8inf", 130, 70, 40, "e5m2", 1.0, False, 86, "uniform", lo=0.5, hi=1.0)
    A, B = si.make_operands(w)
    A[7, :] = np.uint8(0x3C)          # 1.0 across row 7
    A[7, 2] = np.uint8(0x7C)          # +inf
    B[11, 2] = np.uint8(0x00)         # 0 * inf -> NaN in column 11
    B[12, 2] = np.uint8(0xBC)         # -1 * inf -> -inf in column 12
    out = logical(run_tg(w, A, B), w)
    row = out[7]
    assert np.isnan(row[11]) and row[12] == -np.inf
    assert np.all(np.isposinf(np.delete(row, [11, 12])))
    assert np.all(np.isfinite(np.delete(out, 7, axis=0)))


@pytest.mark.parametrize("name", ["f8_e4m3_8192", "f8_e5m2_8192"])
def test_fp8_8192_full(name):
    check_full(si.WORKLOADS[name])
