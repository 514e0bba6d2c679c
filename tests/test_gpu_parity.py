"""CUDA path against the oracle, element by element, through the C ABI.

Every workload of the pages' configurations runs at its full size with the
planner's own choice (the launch configuration the benchmark times) and is
compared on every output element; smaller problems sweep the ragged edges,
every compiled tile configuration, both producers, both operand roles and
the special cases (K = 0, alpha = 0, ReLU of all-negative sums, NaN inputs).
"""

from __future__ import annotations

import numpy as np
import pytest

import seeded_inputs as si
from gemm_harness import assert_within, check_full, logical, run_tg

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_gemm_epilogue_gb300 as tg

    tg.build()
    tg.load()


@pytest.mark.parametrize("name", ["c1_bf16_65x97x73", "c2_tf32_256x128x512"])
def test_small_configs_full(name):
    check_full(si.WORKLOADS[name], repeats=2)


def _edge_cases():
    sizes = [1, 2, 15, 16, 17, 63, 64, 65, 127, 128, 129, 255, 256, 257]
    rng = np.random.default_rng(7)
    picks = {(s, s, s) for s in sizes}
    while len(picks) < 90:
        picks.add(tuple(int(x) for x in rng.choice(sizes, 3)))
    return sorted(picks)


@pytest.mark.parametrize("M,N,K", _edge_cases())
def test_edge_sweep_bf16(M, N, K):
    w = si.Workload(f"edge{M}x{N}x{K}", M, N, K, "bf16", 1.5, True, 100 + M + 7 * N + 13 * K,
                    "uniform")
    check_full(w)


@pytest.mark.parametrize("dtype", ["fp16", "tf32"])
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (129, 65, 33), (257, 255, 129), (17, 300, 70)])
def test_edge_sweep_other_types(dtype, M, N, K):
    w = si.Workload(f"edge_{dtype}", M, N, K, dtype, -0.75, dtype == "fp16", 5 + M + N + K,
                    "uniform")
    check_full(w)


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "tf32"])
@pytest.mark.parametrize("block_n", [64, 128, 256])
@pytest.mark.parametrize("producer", [1, 2])
def test_every_config(dtype, block_n, producer):
    """Each compiled tile configuration and both producers on a ragged
    problem spanning several tiles in M, N and K."""
    w = si.Workload("cfg", 300, 520, 200, dtype, 1.25, True, 17, "uniform", lda=208, ldb=216,
                    ldc=304)
    check_full(w, opts={"block_n": block_n, "producer": producer, "cta_pair": 1})


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("block_n", [128, 256])
@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (129, 300, 64), (513, 1000, 1000), (1, 17, 8)])
def test_cta_pair_configs(dtype, block_n, M, N, K):
    """CTA-pair tiles (256 rows over a 2-CTA cluster, cta_group::2 MMA):
    ragged rows that leave the peer's half partly or wholly outside M."""
    w = si.Workload("pair", M, N, K, dtype, 0.75, True, 19 + M + N, "uniform", ldc=M + 3)
    check_full(w, opts={"cta_pair": 2, "block_n": block_n})


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("block_n", [128, 256])
@pytest.mark.parametrize("M,N,K", [(600, 1100, 520), (257, 500, 64), (1000, 1800, 2048), (90, 700, 128)])
def test_multicast_clusters(dtype, block_n, M, N, K):
    """Two CTA pairs per cluster sharing their A rows by TMA multicast; odd
    N-block counts give the second pair a tile wholly outside N."""
    w = si.Workload("mc", M, N, K, dtype, 1.25, True, 91 + M + N, "uniform", ldc=M + 7)
    check_full(w, opts={"cta_pair": 2, "multicast": 2, "block_n": block_n, "swap_ab": 1},
               repeats=2)


def test_multicast_persistent_swapped_and_batched():
    from gemm_harness import check_batched

    w = si.Workload("mc_p", 1300, 1500, 704, "bf16", 1.0, True, 92, "normal")
    for g in (4, 8, 12):
        check_full(w, opts={"cta_pair": 2, "multicast": 2, "max_ctas": g, "raster_group": 2})
    # Swapped roles: role-space N is the original M (300 -> two N blocks).
    ws = si.Workload("mc_s", 300, 2000, 512, "fp16", 1.0, False, 93, "uniform", ldc=304)
    check_full(ws, opts={"cta_pair": 2, "multicast": 2, "swap_ab": 2})
    wb = si.Workload("mc_b", 500, 700, 1024, "bf16", -1.0, True, 94, "uniform")
    check_batched(wb, 3, "bf16", opts={"cta_pair": 2, "multicast": 2})


def test_cta_pair_persistent_and_swapped():
    w = si.Workload("pair_persist", 1100, 900, 320, "bf16", 1.0, True, 37, "normal")
    for g in (2, 6):
        check_full(w, opts={"cta_pair": 2, "max_ctas": g, "raster_group": 2})
    ws = si.Workload("pair_swap", 100, 2000, 256, "fp16", 1.0, False, 38, "uniform", ldc=104)
    check_full(ws, opts={"cta_pair": 2, "swap_ab": 2})


@pytest.mark.parametrize("M,N,K,max_ctas,split_k,segs", [
    (300, 600, 1024, 8, 8, 2),     # 6 pair tiles on 4 pairs: 2 tail tiles x 2 segments
    (1100, 200, 2104, 8, 8, 4),    # 5 tiles on 4 pairs: 1 tail tile x 4 segments (ragged K)
    (1100, 200, 2104, 8, 3, 3),    # at most 3 segments
    (700, 300, 1000, 4, 8, 1),     # 6 tiles on 2 pairs: none left over -> whole tiles only
    (1100, 260, 1024, 16, 8, 2),   # 16 K blocks allow at most 2 segments of >= 8 blocks
    (1100, 200, 2104, 8, 1, 1),    # split off
    (500, 500, 2048, 0, 0, 4),     # default split: 4 tiles on all pairs -> 4 segments of 8 blocks
])
def test_split_k_tail(M, N, K, max_ctas, split_k, segs):
    """The last, partial wave of pair tiles is cut into K segments whose
    partial sums are added by the last segment in a fixed order: within the
    tolerance, deterministic over repeated calls, flags left clean."""
    import dense_gemm_epilogue_gb300 as tg

    w = si.Workload("split", M, N, K, "bf16", 1.25, True, 53 + M + K, "normal", ldc=M + 5)
    opts = {"cta_pair": 2, "block_n": 256, "max_ctas": max_ctas, "split_k": split_k}
    lda, ldb, ldc = w.strides
    plan = tg.tg_plan(M, N, K, None, lda, None, ldb, None, ldc, "bf16", opts)
    assert plan["split_segs"] == segs
    assert (plan["split_tiles"] > 0) == (segs > 1)
    check_full(w, opts=opts, repeats=3)


@pytest.mark.parametrize("swap", [1, 2])
@pytest.mark.parametrize("M,N", [(64, 1000), (200, 333), (5, 700)])
def test_swap_roles(swap, M, N):
    w = si.Workload("swap", M, N, 150, "bf16", 0.5, True, 23, "uniform", ldc=M + 4)
    check_full(w, opts={"swap_ab": swap})


@pytest.mark.parametrize("prefetch_k", [4, 8, 16])
def test_l2_prefetch_option(prefetch_k):
    """Single-CTA TMA tiles with the A-role L2 burst prefetch (skinny N)."""
    w = si.Workload("prefetch", 2000, 64, 1500, "bf16", 1.0, True, 57, "uniform", lda=1512,
                    ldb=1504, ldc=2008)
    check_full(w, opts={"cta_pair": 1, "prefetch_k": prefetch_k})


def test_swap_scalar_store_unaligned_ldc():
    w = si.Workload("swap_ldc", 33, 900, 77, "fp16", 1.0, False, 29, "uniform", ldc=35)
    check_full(w, opts={"swap_ab": 2})


def test_persistent_multiple_tiles_per_cta():
    """A grid smaller than the tile count: each CTA walks several tiles and
    both tensor-memory accumulators are reused."""
    w = si.Workload("persist", 1000, 1100, 300, "bf16", 1.0, True, 31, "normal")
    for g in (1, 3, 7):
        check_full(w, opts={"max_ctas": g, "raster_group": 2, "cta_pair": 1})


def test_k_zero_gives_epilogue_of_zero():
    w = si.Workload("k0", 70, 90, 0, "bf16", 2.0, True, 1, "uniform", lda=1, ldb=1, ldc=72)
    check_full(w)


def test_alpha_zero_and_negative_products():
    base = si.Workload("az", 200, 180, 96, "bf16", 0.0, True, 41, "uniform")
    check_full(base)
    A, B = si.make_operands(si.with_shape(base, lo=0.0, hi=1.0))
    # A >= 0, B <= 0 (flip B's sign bit): with alpha > 0 every sum is <= 0.
    Bn = B.copy()
    Bn[:, : base.K] |= np.uint16(0x8000)
    w = si.with_shape(base, alpha=1.0)
    out = run_tg(w, A, Bn)
    assert np.all(logical(out, w) == 0.0) and not np.any(np.signbit(logical(out, w)))
    # Negative alpha flips which entries survive.
    wn = si.with_shape(base, alpha=-1.0)
    outn = run_tg(wn, A, Bn)
    assert np.all(logical(outn, wn) > 0.0)


def test_nan_input_propagates_through_relu():
    w = si.Workload("nan", 130, 70, 40, "bf16", 1.0, True, 43, "uniform")
    A, B = si.make_operands(w)
    A[5, 3] = np.uint16(0x7FC0)
    out = logical(run_tg(w, A, B), w)
    assert np.all(np.isnan(out[5, :]))
    assert not np.any(np.isnan(np.delete(out, 5, axis=0)))


def test_repeated_calls_bitwise_identical():
    w = si.Workload("rep", 513, 700, 1000, "bf16", 1.0, True, 47, "normal")
    check_full(w, repeats=3)


def test_invalid_arguments_launch_nothing():
    import torch
    import dense_gemm_epilogue_gb300 as tg

    D = torch.full((10, 10), 7.0, device="cuda")
    A = torch.zeros((10, 10), dtype=torch.int16, device="cuda")
    assert tg.tg_gemm(10, 10, 10, 1.0, A, 9, A, 10, D, 10, "bf16", True) == tg.TG_ERR_INVALID_VALUE
    assert tg.tg_gemm(10, 10, 10, 1.0, A, 10, A, 10, D, 9, "bf16", True) == tg.TG_ERR_INVALID_VALUE
    assert tg.tg_gemm(10, 10, 10, 1.0, None, 10, A, 10, D, 10, "bf16", True) == \
        tg.TG_ERR_INVALID_VALUE
    torch.cuda.synchronize()
    assert torch.all(D == 7.0)


def test_wait_timeout_selftest_reports_status():
    """A bounded wait on a barrier nothing completes runs out, records its
    site and returns; the context stays usable."""
    import torch
    import dense_gemm_epilogue_gb300 as tg

    assert tg.tg_check_device_status()[0] == tg.TG_OK
    assert tg.tg_selftest_wait_timeout(2_000_000) == tg.TG_OK
    st, where = tg.tg_check_device_status()
    assert st == tg.TG_ERR_DEVICE_TIMEOUT and where == 7
    assert tg.tg_check_device_status()[0] == tg.TG_OK      # cleared
    x = torch.ones(4, device="cuda")
    assert float((x * 2).sum()) == 8.0                      # context still fine
    check_full(si.WORKLOADS["c1_bf16_65x97x73"])


@pytest.mark.parametrize("name", ["c5a_bf16_16384x64x4096", "c5b_bf16_64x16384x4096",
                                  "c5c_bf16_8191x4097x1000", "c3_fp16_4096"])
def test_large_configs_full(name):
    check_full(si.WORKLOADS[name])


def test_headline_8192_full():
    """The 8192^3 BF16 + ReLU workload, every element against the oracle."""
    check_full(si.WORKLOADS["c4_bf16_8192"])


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "e4m3"])
@pytest.mark.parametrize("M,N,K", [(300, 520, 1024), (1100, 1300, 640), (257, 4000, 512),
                                   (1, 17, 64), (2000, 2000, 2048)])
def test_dynamic_schedule(dtype, M, N, K):
    """One 2-CTA cluster per tile; running clusters take over the tiles of
    clusters not yet started (cluster launch control).  Every tile exactly
    once: full parity, bitwise repeatable."""
    w = si.Workload("dyn", M, N, K, dtype, 1.25, True, 61 + M + N, "normal", ldc=M + 5)
    check_full(w, opts={"schedule": 2}, repeats=3)


def test_dynamic_schedule_swapped_batched_narrow():
    from gemm_harness import check_batched

    ws = si.Workload("dyn_s", 100, 3000, 512, "bf16", 1.0, False, 62, "uniform", ldc=104)
    check_full(ws, opts={"schedule": 2, "swap_ab": 2})
    wb = si.Workload("dyn_b", 600, 700, 1024, "fp16", -1.0, True, 63, "normal")
    check_batched(wb, 3, "bf16", opts={"schedule": 2})
    check_batched(wb, 2, "f32", share_a=True, opts={"schedule": 2, "block_n": 128})


@pytest.mark.parametrize("dtype,opts", [("bf16", {"cta_pair": 1}), ("bf16", None), ("e4m3", None),
                                        ("tf32", None)])
def test_long_k_accumulation(dtype, opts):
    """K = 131072 (2048 BF16 K blocks; 1024 for FP8, 4096 for TF32): every
    stage barrier wraps its phase hundreds of times within one tile."""
    w = si.Workload("longk", 256, 384, 131072, dtype, 0.25, True, 81, "uniform", ldc=259)
    check_full(w, opts=opts)


def test_many_ragged_tiles_sampled():
    """A 24577 x 24575 output (9312 CTA-pair tiles, 123 waves, ragged in both
    dimensions) against the oracle on sampled entries: every edge row and
    column plus 20000 random elements; D's padding untouched."""
    import oracle
    from gemm_harness import assert_within

    w = si.Workload("many", 24577, 24575, 512, "bf16", 1.0, True, 82, "normal", ldc=24580)
    lda, ldb, ldc = w.strides
    A, B = si.make_operands(w)
    D0 = si.make_output(w)
    out = run_tg(w, A, B, D0)
    rng = np.random.default_rng(83)
    I = np.concatenate([rng.integers(0, w.M, 20000), np.full(w.N, w.M - 1), np.arange(w.M) % w.M])
    J = np.concatenate([rng.integers(0, w.N, 20000), np.arange(w.N), np.full(w.M, w.N - 1)])
    ref, scale = oracle.gemm_entries(w.M, w.N, w.K, w.alpha, A, lda, B, ldb, w.dtype, w.relu, I, J)
    got = out[J, I]
    assert_within(got, ref, scale, w.dtype, w.name)
    assert np.array_equal(out[:, w.M:].view(np.uint32), D0[:, w.M:].view(np.uint32))


def test_cross_check_against_torch_matmul():
    """An extra signal beside the oracle: torch.matmul (cuBLAS, FP32, no TF32)
    on the same buffers, D^T = relu(alpha * B_t A_t^T), within the same bound."""
    import torch

    w = si.Workload("xcheck", 1000, 1500, 2048, "bf16", 0.5, True, 800, "normal", ldc=1004)
    lda, ldb, ldc = w.strides
    A, B = si.make_operands(w)
    D = run_tg(w, A, B, si.make_output(w))
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        At = torch.from_numpy(A.view(np.int16)).cuda().view(torch.bfloat16)[:, : w.K].float()
        Bt = torch.from_numpy(B.view(np.int16)).cuda().view(torch.bfloat16)[:, : w.K].float()
        ref = torch.relu(w.alpha * (Bt @ At.T))                       # (N, M)
        scale = abs(w.alpha) * (Bt.abs() @ At.abs().T)
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    got = torch.from_numpy(np.ascontiguousarray(D[:, : w.M])).cuda()
    err = (got - ref).abs()
    assert bool((err <= 2.0 ** -7 * scale + 1e-6).all()), float(err.max())


def test_rotated_k_order_one_wave():
    """One wave of single-CTA tiles, each walking its K blocks from its own
    offset (K ragged against the stage, so the wrap crosses the partial last
    block), TMA and plain loads; bitwise repeatable."""
    import dense_gemm_epilogue_gb300 as tg

    for producer, lda in ((1, 2056), (2, 2049)):
        w = si.Workload("rot", 1000, 500, 2049, "bf16", 1.0, True, 91 + producer, "normal",
                        lda=lda, ldb=lda, ldc=1003)
        opts = {"cta_pair": 1, "block_n": 128, "split_k": 1, "producer": producer}
        p = tg.tg_plan(w.M, w.N, w.K, None, lda, None, lda, None, w.ldc, w.dtype, opts)
        assert p["k_rotate"] == 1 and p["tiles"] <= p["grid"]
        check_full(w, opts=opts, repeats=2)
