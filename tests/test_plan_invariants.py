"""Properties every plan must have, over a seeded sweep of problem shapes,
operand types, strides and SM counts (host only: tg_plan with an SM count
touches no CUDA).  The named cases in test_abi_host.py pin particular
choices; this file checks that no shape leads the planner into a plan the
kernels cannot run: a grid larger than the device or not made of whole
clusters, tiles that do not cover the output, a K split where none is
allowed, a tensor-memory or shared-memory budget out of range."""

from __future__ import annotations

import numpy as np
import pytest

SMEM_LIMIT = 232448
ELEM = {"bf16": 2, "fp16": 2, "tf32": 4, "e4m3": 1, "e5m2": 1}
BASE = 1 << 20          # a 1 MB-aligned fake device address (planning reads only its alignment)


@pytest.fixture(scope="module")
def tg():
    import dense_gemm_epilogue_gb300 as tg

    tg.build()
    tg.load()
    return tg


def cdiv(a, b):
    return -(-a // b)


def shapes(seed=2024, n=1500):
    """Problem sizes in four regimes: log-uniform over 1 .. 20000 (tiny, odd
    and skinny shapes), large (M, N >= 512 and K >= 256: CTA-pair tiles,
    multicast clusters), mid-sized with long K (fewer tiles than pairs: K
    splits) and skinny (one of M, N below 128: swapped roles, stream-K);
    tight, padded or TMA-illegal strides."""
    rng = np.random.default_rng(seed)
    out = []
    for q in range(n):
        regime = q % 4
        if regime == 0:
            M, N, K = (int(round(10 ** rng.uniform(0, 4.3))) for _ in range(3))
        elif regime == 1:
            M, N = (int(round(10 ** rng.uniform(2.7, 4.3))) for _ in range(2))
            K = int(round(10 ** rng.uniform(2.4, 4.6)))
        elif regime == 2:
            M, N = (int(round(10 ** rng.uniform(2.3, 3.3))) for _ in range(2))
            K = int(round(10 ** rng.uniform(3.5, 4.8)))
        else:
            M = int(rng.integers(1, 128))
            N = int(round(10 ** rng.uniform(2.1, 4.3)))
            K = int(round(10 ** rng.uniform(1.5, 4.8)))
            if rng.random() < 0.5:
                M, N = N, M
        dtype = str(rng.choice(list(ELEM)))
        per16 = 16 // ELEM[dtype]                   # elements per 16 bytes
        mode = str(rng.choice(["aligned", "aligned", "aligned_pad", "tight", "odd"]))
        ld = {"aligned": cdiv(K, per16) * per16, "aligned_pad": cdiv(K, per16) * per16 + per16,
              "tight": K, "odd": K + 1}[mode]
        out.append((M, N, K, dtype, ld, ld, M + int(rng.choice([0, 8, 1])),
                    int(rng.choice([152, 152, 148, 132, 64, 16, 7, 2, 1]))))
    return out


def check_plan(p, M, N, K, dtype, lda, ldb, ldc, sms):
    e = ELEM[dtype]
    nkb = cdiv(K, 128 // e)
    assert p["block_k"] == 128 // e
    # Roles: a short M with a long N runs swapped.
    swap = M < 128 and N >= 128 and N >= 2 * M
    assert p["swap_ab"] == int(swap)
    mk, nk = (N, M) if swap else (M, N)
    # Producer: TMA exactly when bases and row strides are 16-byte multiples.
    legal = (lda * e) % 16 == 0 and (ldb * e) % 16 == 0
    assert p["producer"] == (1 if legal else 2)
    # Tile shape and coverage.
    pair = p["cta_pair"] == 1
    assert p["block_m"] == (256 if pair else 128)
    assert p["block_n"] in ((128, 256) if pair else (64, 128, 256))
    mc = p["multicast"]
    assert mc == (0 if not pair else mc) and (mc in (1, 2) if pair else mc == 0)
    nblocks = cdiv(nk, p["block_n"])
    assert p["tiles"] == cdiv(mk, p["block_m"]) * cdiv(nblocks, max(mc, 1))
    assert 1 <= p["raster_group"] <= cdiv(mk, p["block_m"])
    if pair:
        assert dtype != "tf32" and legal and nkb >= 8
        if mc == 2:
            assert nkb <= 32 and nblocks >= 2
    # Grid: whole clusters, never more CTAs than SMs (at least one cluster).
    g = p["grid"]
    assert g >= 1
    if pair:
        assert g % (2 * mc) == 0 and g <= max(sms - sms % (2 * mc), 2 * mc)
    else:
        assert g <= sms
        if not p["stream_k"]:
            assert g == min(p["tiles"], sms)
    # K splits: segments of at least 8 K blocks, only on pair tiles with one
    # pair per cluster; stream-K only on single-CTA tiles.
    segs, st = p["split_segs"], p["split_tiles"]
    assert segs >= 1 and 0 <= st <= p["tiles"]
    if segs > 1:
        # The last round's R = tiles mod pairs tiles, S segments each, fit
        # on the round's pairs.
        assert pair and mc == 1 and segs <= 8 and segs <= nkb // 8
        assert st == p["tiles"] % (g // 2) and st >= 1 and st * segs <= g // 2
    else:
        assert st == 0
    if p["stream_k"]:
        assert not pair and segs == 1
        assert g <= p["tiles"] * nkb // 8 or g == 1
    # Per-CTA budgets the kernels were compiled for.
    assert 0 < p["smem_bytes"] <= SMEM_LIMIT
    t = p["tmem_cols"]
    assert 32 <= t <= 512 and t & (t - 1) == 0
    assert p["threads"] % 32 == 0 and 0 < p["threads"] <= 1024
    assert p["stages"] >= 2
    if p["vector_store"]:
        assert swap
    # Alternating K order: 16-bit pair tiles under tickets, and nowhere else.
    assert p["k_snake"] == int(pair and p["schedule"] == 4 and dtype in ("bf16", "fp16"))
    if p["k_rotate"]:
        assert not pair and not p["stream_k"] and p["tiles"] <= g


def test_plans_over_a_sweep_of_shapes(tg):
    seen = {"pair": 0, "multicast": 0, "split": 0, "stream_k": 0, "swap": 0, "plain": 0,
            "single": 0, "vector": 0}
    for M, N, K, dtype, lda, ldb, ldc, sms in shapes():
        p = tg.tg_plan(M, N, K, BASE, lda, BASE, ldb, BASE, ldc, dtype, None, sms)
        check_plan(p, M, N, K, dtype, lda, ldb, ldc, sms)
        # The planner is a pure function of its arguments.
        assert tg.tg_plan(M, N, K, BASE, lda, BASE, ldb, BASE, ldc, dtype, None, sms) == p
        seen["pair"] += p["cta_pair"]
        seen["single"] += 1 - p["cta_pair"]
        seen["multicast"] += p["multicast"] == 2
        seen["split"] += p["split_segs"] > 1
        seen["stream_k"] += p["stream_k"]
        seen["swap"] += p["swap_ab"]
        seen["plain"] += p["producer"] == 2
        seen["vector"] += p["vector_store"]
    # The sweep reaches every kind of plan, so the checks above are not vacuous.
    assert all(v >= 5 for v in seen.values()), seen


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (1, 20000, 7), (20000, 1, 7), (128, 128, 64),
                                   (255, 257, 8 * 64), (256, 256, 7 * 64), (8191, 4097, 1000)])
@pytest.mark.parametrize("sms", [152, 2, 1])
def test_plans_at_boundaries(tg, M, N, K, sms):
    for dtype in ELEM:
        p = tg.tg_plan(M, N, K, BASE, K, BASE, K, BASE, M, dtype, None, sms)
        check_plan(p, M, N, K, dtype, K, K, M, sms)


def test_grid_cap_is_respected(tg):
    """max_ctas bounds the persistent grid (rounded down to whole clusters, at
    least one cluster) without changing what the tiles cover."""
    rng = np.random.default_rng(7)
    for M, N, K, dtype, lda, ldb, ldc, sms in shapes(seed=99, n=400):
        cap = int(rng.integers(1, 200))
        p = tg.tg_plan(M, N, K, BASE, lda, BASE, ldb, BASE, ldc, dtype, {"max_ctas": cap}, sms)
        check_plan(p, M, N, K, dtype, lda, ldb, ldc, min(sms, cap))
        if p["cta_pair"]:
            cl = 2 * p["multicast"]
            assert p["grid"] <= cl * max(1, min(sms, cap) // cl)
        else:
            assert p["grid"] <= min(sms, cap)


def test_block_scaled_plans_over_a_sweep(tg):
    """The block-scaled planner: CTA-pair tiles 256 x 128 or 256 x 256 over
    all pairs of the device (fewer when there are fewer tiles); TMA for
    strides of 16-byte multiples, the plain-load producer on 256 x 128 tiles
    for the others (forcing TMA on them, or odd FP4 rows, are refused)."""
    rng = np.random.default_rng(31)
    for M, N, K, dtype, _, _, ldc, sms in shapes(seed=5, n=600):
        kind = str(rng.choice(["e4m3", "e5m2", "e2m1", "nvf4"]))
        fp4 = kind in ("e2m1", "nvf4")
        if fp4:
            K += K & 1                                  # packed FP4: whole bytes per row
        per16 = 32 if fp4 else 16                       # elements per 16 bytes
        ld = cdiv(K, per16) * per16 + per16 * int(rng.integers(0, 2))
        p = tg.tg_plan_mx(M, N, K, ld, ld, ldc, kind, None, sms)
        swap = M < 128 and N >= 128 and N >= 2 * M
        mk, nk = (N, M) if swap else (M, N)
        assert p["swap_ab"] == int(swap) and p["cta_pair"] == 1 and p["producer"] == 1
        assert p["block_m"] == 256 and p["block_n"] in (128, 256)
        assert p["block_k"] == (256 if fp4 else 128)
        assert p["tiles"] == cdiv(mk, 256) * cdiv(nk, p["block_n"])
        assert p["grid"] == 2 * min(p["tiles"], max(1, sms // 2))
        assert 1 <= p["raster_group"] <= cdiv(mk, 256)
        assert 0 < p["smem_bytes"] <= SMEM_LIMIT and p["stages"] >= 2
        t = p["tmem_cols"]
        assert 32 <= t <= 512 and t & (t - 1) == 0
        assert p["threads"] % 32 == 0 and p["threads"] <= 1024
        # A stride that is not a multiple of 16 bytes: plain loads, four more warps.
        bad = ld + (2 if fp4 else 1)
        q = tg.tg_plan_mx(M, N, K, bad, ld, ldc, kind, None, sms)
        assert q["producer"] == 2 and q["block_n"] == 128
        assert q["threads"] == p["threads"] + 128 and q["tiles"] == cdiv(mk, 256) * cdiv(nk, 128)
        with pytest.raises(tg.TgError):
            tg.tg_plan_mx(M, N, K, bad, ld, ldc, kind, {"producer": 1}, sms)
