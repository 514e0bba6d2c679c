"""The seeded input generator (host only, no GPU): its FP8 rounding, its
counter-based SplitMix64 stream against the published sequence, and the
distributions it draws.

The FP8 codes it writes must be the nearest representable values (ties to the
even code, saturating at the largest finite value); checked by brute force over
all 256 codes, decoded by the float16 re-encoding in ``oracle_pin_checks``.
"""

import numpy as np
import pytest

import seeded_inputs as si
from oracle_pin_checks import e4m3_by_fp16, e5m2_by_fp16

DECODE = {"e4m3": e4m3_by_fp16, "e5m2": e5m2_by_fp16}


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_codes_round_trip(fmt):
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    vals = DECODE[fmt](codes)
    fin = np.isfinite(vals)
    back = si.f32_to_fp8_bits(vals[fin].astype(np.float32), fmt)
    assert np.array_equal(back, codes[fin])


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_nearest_by_brute_force(fmt):
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    table = DECODE[fmt](codes)
    fin = np.isfinite(table)
    tv, tc = table[fin], codes[fin]
    top = np.max(tv)
    x = si.normal_f32(9, 0, 4000, 3.0 if fmt == "e4m3" else 50.0)
    x = np.concatenate([x, np.float32([0.0, -0.0, 1e-9, 2 * top, -2 * top])])
    got = si.f32_to_fp8_bits(x, fmt)
    for v, g in zip(x.astype(np.float64), got):
        c = min(max(v, -top), top)
        d = np.abs(tv - c)
        best = np.flatnonzero(d == d.min())
        if v != 0:
            best = best[np.signbit(tv[best]) == np.signbit(v)]
        if best.size > 1:      # a tie: the even code
            best = best[tc[best] % 2 == 0]
        assert g in tc[best], (fmt, v, g, tc[best])


def test_fp8_nan_and_signed_zero():
    for fmt in ("e4m3", "e5m2"):
        c = si.f32_to_fp8_bits(np.float32([np.nan, -0.0, 0.0]), fmt)
        assert np.isnan(DECODE[fmt](c[:1]))[0]
        assert c[1] == 0x80 and c[2] == 0x00


def test_e2m1_nearest_by_brute_force_and_packing():
    from oracle_pin_checks import E2M1_TABLE

    table = np.array(E2M1_TABLE)
    x = np.concatenate([si.normal_f32(11, 0, 3000, 2.5),
                        np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.5, 100.0, -0.25, -5.0])])
    codes = si.f32_to_e2m1_codes(x)
    for v, c in zip(x.astype(np.float64), codes):
        cv = min(max(v, -6.0), 6.0)
        d = np.abs(table - cv)
        best = np.flatnonzero(d == d.min())
        if v != 0:
            best = best[np.signbit(table[best]) == np.signbit(v)]
        if best.size > 1:
            best = best[best % 2 == 0]
        assert c in best, (v, c, best)
    packed = si.pack_e2m1(np.arange(16, dtype=np.uint8))
    assert list(packed) == [0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE]


def test_splitmix64_published_sequence():
    """SplitMix64 (Steele, Lea and Flood; Vigna's reference implementation):
    from state 1234567 the first five outputs are these published values."""
    gamma = 0x9E3779B97F4A7C15
    states = np.array([(1234567 + (i + 1) * gamma - gamma) % (1 << 64) for i in range(5)],
                      dtype=np.uint64)
    got = [int(v) for v in si.splitmix64(states)]
    assert got == [6457827717110365317, 3203168211198807973, 9817491932198370423,
                   4593380528125082431, 16408922859458223821]


def test_draws_are_positional_and_reproducible():
    """Element i always gets the same draw, whatever the count asked for (so a
    sample of a workload sees the full workload's entries), and the streams of
    one seed and the seeds of one stream differ."""
    n = si.CHUNK + 5
    for f in (lambda c: si.uniform_f32(3, 0, c, -1.0, 1.0), lambda c: si.normal_f32(3, 0, c)):
        big, small = f(n), f(1000)
        assert np.array_equal(big[:1000], small)
        assert np.array_equal(f(1000), small)
    assert not np.array_equal(si.uniform_f32(3, 0, 64, 0.0, 1.0), si.uniform_f32(3, 1, 64, 0.0, 1.0))
    assert not np.array_equal(si.uniform_f32(3, 0, 64, 0.0, 1.0), si.uniform_f32(4, 0, 64, 0.0, 1.0))


def test_uniform_grid_and_moments():
    """Uniform entries lie on the 2^-24 grid of [lo, hi) and have the mean and
    variance of U[lo, hi) within six standard errors; the A and B streams are
    uncorrelated."""
    n = 1 << 20
    u = si.uniform01(0, 0, 0, n)
    assert u.min() >= 0.0 and u.max() < 1.0
    assert np.array_equal(u * 2.0 ** 24, np.floor(u * 2.0 ** 24))
    for lo, hi in ((-1.0, 1.0), (0.0, 1.0)):
        x = si.uniform_f32(1, 0, n, lo, hi).astype(np.float64)
        assert x.min() >= lo and x.max() < hi
        var = (hi - lo) ** 2 / 12
        assert abs(x.mean() - (lo + hi) / 2) < 6 * np.sqrt(var / n)
        assert abs(x.var() - var) < 6 * var * np.sqrt(0.8 / n)     # var of (x-m)^2 is 0.8 var^2
    a = si.uniform_f32(4, si.STREAM_A, n, -1.0, 1.0).astype(np.float64)
    b = si.uniform_f32(4, si.STREAM_B, n, -1.0, 1.0).astype(np.float64)
    assert abs(np.corrcoef(a, b)[0, 1]) < 6 / np.sqrt(n)


def test_normal_moments_and_tails():
    """Box-Muller entries: mean 0, variance 1, no skew, kurtosis 3 (each within
    six standard errors), tail masses of N(0, 1) beyond 2 and 3, and the scale
    factor applied exactly."""
    n = 1 << 21
    z = si.normal_f32(3, 0, n).astype(np.float64)
    assert abs(z.mean()) < 6 / np.sqrt(n)
    assert abs(z.var() - 1.0) < 6 * np.sqrt(2.0 / n)
    assert abs(np.mean(z ** 3)) < 6 * np.sqrt(15.0 / n)
    assert abs(np.mean(z ** 4) - 3.0) < 6 * np.sqrt(96.0 / n)
    for t, p in ((2.0, 0.0455002638963584), (3.0, 0.0026997960632602)):
        frac = np.mean(np.abs(z) > t)
        assert abs(frac - p) < 6 * np.sqrt(p * (1 - p) / n)
    # Scaled draws are the unscaled ones times the factor (each side rounded
    # once to FP32 from a double, so within two FP32 half-ulps).
    z01 = si.normal_f32(3, 0, 4096, 0.1).astype(np.float64)
    z1 = si.normal_f32(3, 0, 4096).astype(np.float64)
    assert np.all(np.abs(z01 - 0.1 * z1) <= 2.0 ** -22 * np.abs(z01))
