"""The kernels' work decomposition, restated on the host and checked for
exact coverage (no GPU).

The kernels map a linear tile index to an output tile by a grouped raster
(`tile_coords` in csrc/tg_kernel.cuh), hand whole tiles to persistent CTAs or
pairs, cut the last partial wave of CTA-pair tiles into K segments
(`make_unit_plan` / `decode_unit` in csrc/tg_kernel_pair.cuh), or give each
CTA a contiguous share of all (tile, K block) iterations (stream-K,
`TileUnits` in csrc/tg_kernel.cuh).  The functions below restate those
rules in Python; the tests drive them with the planner's own choices
(tg_plan) and check that every output tile, and every K block of it, is
computed exactly once, that the unit that finishes a cut tile only waits on
work dispatched before it, and that workspace slots and flags stay inside
what the host allocates.
"""

from __future__ import annotations

import numpy as np
import pytest

BASE = 1 << 20


@pytest.fixture(scope="module")
def tg():
    import dense_gemm_epilogue_gb300 as tg

    tg.build()
    tg.load()
    return tg


def cdiv(a, b):
    return -(-a // b)


# ---------------------------------------------------------------- restatements

def tile_coords(t, num_m_blocks, num_n_blocks, group):
    """Grouped raster: groups of `group` M blocks; inside a group, M fastest."""
    per_group = group * num_n_blocks
    g = t // per_group
    first_m = g * group
    gsz = min(num_m_blocks - first_m, group)
    r = t - g * per_group
    return first_m + r % gsz, r // gsz


def stream_k_units(cta, grid, tiles, nkb):
    """CTA `cta`'s share [cta*I/G, (cta+1)*I/G) of I = tiles*nkb iterations,
    cut at tile boundaries into (tile, k0, k1) units."""
    total = tiles * nkb
    pos, end = total * cta // grid, total * (cta + 1) // grid
    out = []
    while pos < end:
        t = pos // nkb
        k0 = pos - t * nkb
        k1 = min(k0 + (end - pos), nkb)
        out.append((t, k0, k1))
        pos += k1 - k0
    return out


def unit_plan(tiles, pairs, nkb, split_max, ws_tiles):
    """Whole tiles first, then the last R = tiles mod pairs tiles cut into
    S K segments each (S = min(pairs / R, split_max, nkb / 8))."""
    rem, segs = tiles % pairs, 1
    if split_max > 1 and rem > 0:
        s = min(pairs // rem, split_max, nkb // 8)
        if s > 1 and rem * (s - 1) <= ws_tiles:
            segs = s
    whole = tiles - rem if segs > 1 else tiles
    return whole, segs, whole + (tiles - whole) * segs


def decode_unit(u, whole, segs, nkb):
    """Unit u -> (tile, k0, k1, segment, tail index); segment -1: whole tile."""
    if u < whole:
        return u, 0, nkb, -1, 0
    j = u - whole
    tail, seg = j // segs, j % segs
    return whole + tail, seg * nkb // segs, (seg + 1) * nkb // segs, seg, tail


# ---------------------------------------------------------------- tests

@pytest.mark.parametrize("seed", range(4))
def test_raster_is_a_bijection(seed):
    rng = np.random.default_rng(seed)
    for _ in range(200):
        nm, nn = int(rng.integers(1, 70)), int(rng.integers(1, 70))
        group = int(rng.integers(1, nm + 1))
        seen = set()
        for t in range(nm * nn):
            mb, nb = tile_coords(t, nm, nn, group)
            assert 0 <= mb < nm and 0 <= nb < nn
            seen.add((mb, nb))
        assert len(seen) == nm * nn


def shapes(seed, n):
    rng = np.random.default_rng(seed)
    for _ in range(n):
        M, N = (int(round(10 ** rng.uniform(1.5, 4.0))) for _ in range(2))
        K = int(round(10 ** rng.uniform(2.0, 4.8)))
        dtype = str(rng.choice(["bf16", "fp16", "tf32", "e4m3"]))
        per16 = {"bf16": 8, "fp16": 8, "tf32": 4, "e4m3": 16}[dtype]
        yield M, N, K, dtype, cdiv(K, per16) * per16, int(rng.choice([152, 148, 64, 16, 7]))


def test_stream_k_covers_every_iteration_once(tg):
    checked = cut = 0
    for M, N, K, dtype, ld, sms in shapes(11, 600):
        p = tg.tg_plan(M, N, K, BASE, ld, BASE, ld, BASE, M, dtype, {"schedule": 3}, sms)
        tiles, grid = p["tiles"], p["grid"]
        nkb = cdiv(K, p["block_k"])
        assert grid <= sms
        count = np.zeros((tiles, nkb), dtype=np.int64)
        first_units = {}
        for c in range(grid):
            units = stream_k_units(c, grid, tiles, nkb)
            for i, (t, k0, k1) in enumerate(units):
                count[t, k0:k1] += 1
                if k0 > 0:
                    # A contributor is always its CTA's first unit: its
                    # partial goes to the CTA's own slot (one per CTA).
                    assert i == 0
                    first_units[c] = t
        assert (count == 1).all()
        # The owner of a cut tile (the unit with k0 = 0) waits for CTAs
        # c+1 .. c_last, each of which holds the tile as its first unit.
        for c in range(grid):
            units = stream_k_units(c, grid, tiles, nkb)
            for i, (t, k0, k1) in enumerate(units):
                if k0 == 0 and k1 < nkb:
                    # The owner's part is the last unit of its share, so it
                    # never waits on work its own CTA has yet to do.
                    assert i == len(units) - 1
                    c_last = c
                    while c_last + 1 < grid and tiles * nkb * (c_last + 1) // grid < (t + 1) * nkb:
                        c_last += 1
                    assert c_last > c
                    for d in range(c + 1, c_last + 1):
                        assert first_units.get(d) == t
                    cut += 1
        checked += 1
    assert checked == 600 and cut >= 1000


def test_pair_units_cover_every_iteration_once(tg):
    splits = 0
    for M, N, K, dtype, ld, sms in shapes(12, 800):
        if dtype == "tf32":
            continue
        try:
            p = tg.tg_plan(M, N, K, BASE, ld, BASE, ld, BASE, M, dtype, {"cta_pair": 2}, sms)
        except tg.TgError:      # pair tiles refused (fewer than 8 K blocks): skip
            continue
        mc = p["multicast"]
        pairs = p["grid"] // (2 * mc)
        tiles, nkb = p["tiles"], cdiv(K, p["block_k"])
        pairs_max = max(1, sms // (2 * mc))
        ticket = mc == 1 and tiles >= 6 * pairs_max
        assert (p["schedule"] == 4) == ticket
        split_max = 1 if mc != 1 else (8 if tiles < pairs_max else 2)
        ws_tiles = sms // 2                      # what a fresh workspace holds
        whole, segs, units = unit_plan(tiles, pairs, nkb, split_max, ws_tiles)
        # The planner reports the same split the kernel will make.
        assert segs == p["split_segs"]
        assert (tiles - whole if segs > 1 else 0) == p["split_tiles"]
        count = np.zeros((tiles, nkb), dtype=np.int64)
        owner = {}
        if ticket:
            # First unit of each pair static, then claims in order: claim v
            # is unit pairs + v; claims past the end fail, one per pair, and
            # the launch's last claim (v == units - 1) resets the counter.
            assert units >= pairs
            order = list(range(pairs))
            fails = []
            for v in range(units):
                (order if pairs + v < units else fails).append(pairs + v if pairs + v < units else v)
            assert len(fails) == pairs and fails[-1] == units - 1
            dispatch = [(u, u) for u in order]          # (claim order, unit)
        else:
            dispatch = [(u, u) for pair in range(pairs) for u in range(pair, units, pairs)]
        if not ticket and segs == 2 and tiles >= pairs:
            # Static exchange: a tail tile's two segments are consecutive
            # units of the last round, on neighbouring pairs.
            assert whole % pairs == 0
        for rank, u in dispatch:
            t, k0, k1, seg, tail = decode_unit(u, whole, segs, nkb)
            assert k1 - k0 >= min(8, nkb) and k0 < k1
            count[t, k0:k1] += 1
            if seg >= 0:
                owner[(t, seg)] = rank
                if segs == 2:
                    # Exchange halves: partial (tail, segment, CTA half) and
                    # its flag inside the workspace.
                    for half in range(2):
                        assert (tail * 2 + half) * 2 + seg < 4 * ws_tiles
                        assert ((tail * 2 + half) * 2 + seg + 1) * (p["block_n"] // 2) <= \
                            ws_tiles * 2 * 256
                elif seg < segs - 1:
                    pidx = tail * (segs - 1) + seg
                    assert pidx < ws_tiles and pidx * 2 + 1 < 4 * ws_tiles
        assert (count == 1).all()
        if segs > 1:
            splits += 1
            for t in range(whole, tiles):
                us = [owner[(t, s)] for s in range(segs)]
                if ticket:
                    # A tile's segments are consecutive claims: the two sides
                    # of an exchange are handed out one right after the other.
                    assert us == list(range(us[0], us[0] + segs))
                else:
                    # All segments of a tail tile run in the last round, and
                    # the finisher is dispatched after the segments it waits for.
                    assert max(us) - min(us) < pairs
                    assert us[segs - 1] == max(us)
    assert splits >= 20
