"""The seeded input generator's FP8 rounding (host only, no GPU).

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
