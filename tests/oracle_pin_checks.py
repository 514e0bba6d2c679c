"""Checks that pin the oracle to what the definition and the formats fix.

Each ``check_*`` takes an ``oracle.Oracle`` instance and raises
``AssertionError`` on a mismatch.  ``test_oracle_pins.py`` runs them on the
real oracle; ``test_oracle_mutants.py`` runs them on copies of the oracle
with a planted mistake and expects a failure.

None of these checks re-types the oracle's arithmetic: the expected values
come from closed forms, invariants, hand-worked examples, a second decode
written from numpy's own float types, and exact rational arithmetic
(``fractions.Fraction``) on tiny problems.
"""

from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np

import seeded_inputs as si

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- helpers

def bf16_bits_exact(x) -> np.ndarray:
    """float -> bf16 bits for values known to be exactly representable."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exact in bf16"
    return (u >> 16).astype(np.uint16)


def fp16_bits_exact(x) -> np.ndarray:
    f = np.asarray(x, dtype=np.float64)
    h = f.astype(np.float16)
    assert np.array_equal(h.astype(np.float64), f), "value not exact in fp16"
    return h.view(np.uint16)


def fp8_bits_exact(x, dtype) -> np.ndarray:
    """float -> FP8 code for values known to be exactly representable, using
    the float16-based second decode as the table."""
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    table = (e5m2_by_fp16 if dtype == "e5m2" else e4m3_by_fp16)(codes)
    f = np.asarray(x, dtype=np.float64)
    out = np.zeros(f.shape, dtype=np.uint8)
    for idx, v in np.ndenumerate(f):
        hit = np.flatnonzero((table == v) & (np.signbit(table) == np.signbit(v)))
        assert hit.size >= 1, f"{v} not exact in {dtype}"
        out[idx] = hit[0]
    return out


def storage_of(x, dtype):
    if dtype == "bf16":
        return bf16_bits_exact(x)
    if dtype == "fp16":
        return fp16_bits_exact(x)
    if dtype in ("e4m3", "e5m2"):
        return fp8_bits_exact(x, dtype)
    return np.asarray(x, dtype=np.float32)


def second_decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Decode via numpy's own float types (independent of the oracle)."""
    with np.errstate(invalid="ignore"):
        if dtype == "bf16":
            return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        if dtype == "fp16":
            return bits.view(np.float16).astype(np.float64)
    raise ValueError(dtype)


def pack(Alog: np.ndarray, Blog: np.ndarray, dtype: str, lda=None, ldb=None):
    """Logical A (M,K) and B (K,N) -> K-contiguous storage with strides."""
    M, K = Alog.shape
    K2, N = Blog.shape
    assert K == K2
    lda = lda or max(K, 1)
    ldb = ldb or max(K, 1)
    A = np.full((M, lda), si.pad_value(dtype), dtype=si.storage_numpy_dtype(dtype))
    B = np.full((N, ldb), si.pad_value(dtype), dtype=si.storage_numpy_dtype(dtype))
    A[:, :K] = storage_of(Alog, dtype).reshape(M, K)
    B[:, :K] = storage_of(Blog.T, dtype).reshape(N, K)
    return A, lda, B, ldb


def run(orc, Alog, Blog, dtype, alpha, relu, lda=None, ldb=None, **kw):
    A, lda, B, ldb = pack(np.asarray(Alog, float), np.asarray(Blog, float), dtype, lda, ldb)
    M, K = np.asarray(Alog).shape
    N = np.asarray(Blog).shape[1]
    return orc.gemm(M, N, K, alpha, A, lda, B, ldb, dtype, relu, **kw)


def tf32_reference(x: float) -> float:
    """fp32 -> tf32 by the reading 'round to nearest, ties away from zero, 10
    fraction bits, fp32 exponent range', written with frexp and float64
    arithmetic (a second formulation, not the oracle's integer one)."""
    if math.isnan(x) or math.isinf(x) or x == 0.0:
        return x
    a = abs(x)
    if a < 2.0 ** -126:          # fp32 subnormal: fixed rounding position
        unit = 2.0 ** (-126 - 10)
    else:
        _, e = math.frexp(a)     # a = m * 2^e, m in [0.5, 1)
        unit = 2.0 ** (e - 1 - 10)
    q = a / unit                 # exact: a power-of-two scaling
    fl = math.floor(q)
    r = fl + 1 if q - fl >= 0.5 else fl
    y = r * unit
    if y > (2.0 - 2.0 ** -10) * 2.0 ** 127:
        y = math.inf
    return math.copysign(y, x)


# ---------------------------------------------------------------- checks

def check_decode_tables(orc):
    """All 65 536 bf16 and fp16 patterns against numpy's decode."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for dt in ("bf16", "fp16"):
        got = orc.decode(bits, dt)
        want = second_decode(bits, dt)
        nan_g, nan_w = np.isnan(got), np.isnan(want)
        assert np.array_equal(nan_g, nan_w), dt
        ok = ~nan_w
        assert np.array_equal(got[ok], want[ok]), dt
        assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok])), dt


def tf32_probe_patterns(n_random=100_000, seed=11) -> np.ndarray:
    edge = []
    for e in (0, 1, 2, 100, 126, 127, 128, 200, 253, 254, 255):
        for f in (0, 1, 0xFFF, 0x1000, 0x1001, 0x1FFF, 0x2000, 0x3000, 0x7FE000, 0x7FEFFF,
                  0x7FF000, 0x7FFFFF, 0x400000, 0x401000):
            for s in (0, 1):
                edge.append((s << 31) | (e << 23) | f)
    rnd = si.raw_u64(seed, 0, 0, n_random).astype(np.uint64) & np.uint64(0xFFFFFFFF)
    return np.concatenate([np.array(edge, dtype=np.uint64), rnd]).astype(np.uint32)


def check_tf32_narrowing(orc):
    pats = tf32_probe_patterns()
    x = pats.view(np.float32)
    got = orc.decode(x, "tf32")
    with np.errstate(invalid="ignore"):
        x64 = x.astype(np.float64)
    want = np.array([tf32_reference(float(v)) for v in x64])
    nan_g, nan_w = np.isnan(got), np.isnan(want)
    assert np.array_equal(nan_g, nan_w)
    ok = ~nan_w
    assert np.array_equal(got[ok], want[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))


def check_golden(orc):
    with open(os.path.join(GOLDEN, "hand_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        D = run(orc, c["A"], c["B"], c["dtype"], c["alpha"], c["relu"])
        want = np.array(c["D"], dtype=np.float64)
        assert D.shape == want.shape, c["name"]
        assert np.array_equal(D, want), (c["name"], D, want)


def check_identity(orc):
    """A = I (M = K): D = epi(alpha * B) exactly."""
    rng_vals = si.uniform_f32(21, 0, 7 * 9, -1.0, 1.0)
    Bq = second_decode(si.f32_to_bf16_bits(rng_vals), "bf16").reshape(7, 9)
    for alpha, relu in ((1.5, True), (-2.0, True), (0.75, False)):
        D = run(orc, np.eye(7), Bq, "bf16", alpha, relu)
        want = alpha * Bq
        if relu:
            want = np.where(want > 0, want, 0.0)
        assert np.array_equal(D, want)


def check_permutation(orc):
    """A a permutation matrix: row i of D is row p(i) of epi(alpha*B)."""
    p = np.array([3, 0, 4, 1, 2])
    P = np.zeros((5, 5))
    P[np.arange(5), p] = 1.0
    vals = si.uniform_f32(22, 0, 5 * 6, -1.0, 1.0)
    Bq = second_decode(si.f32_to_bf16_bits(vals), "bf16").reshape(5, 6)
    D = run(orc, P, Bq, "bf16", 2.0, False)
    assert np.array_equal(D, 2.0 * Bq[p, :])


def rank1_case():
    u = np.array([1, -3, 2, 5, -1, 7, 4], dtype=float)               # M = 7
    v = np.array([2, -1, 3, -6, 1], dtype=float)                      # N = 5
    s = np.array([0.5, -2, 1, 0.25, 4, -0.125, 2, 1, -1, 8, 0.5])    # K = 11
    t = np.array([2, 0.5, -1, 4, -0.25, 8, 1, -2, 0.5, 0.125, -4])
    return u, v, s, t


def check_rank1(orc):
    """a(i,k) = u_i s_k, b(k,j) = t_k v_j  =>  D = alpha (s.t) u v^T, exact.
    M, N, K all differ, so a transposed operand or output fails."""
    u, v, s, t = rank1_case()
    Alog, Blog = np.outer(u, s), np.outer(t, v)
    st = float(np.dot(s, t))
    for dt in ("bf16", "fp16", "tf32", "e4m3", "e5m2"):
        for alpha, relu in ((1.0, False), (1.5, True), (-0.5, True)):
            D, S = run(orc, Alog, Blog, dt, alpha, relu, with_scale=True)
            want = alpha * st * np.outer(u, v)
            if relu:
                want = np.where(want > 0, want, 0.0)
            assert np.array_equal(D, want), (dt, alpha, relu)
            scale = abs(alpha) * float(np.dot(np.abs(s), np.abs(t))) * np.outer(np.abs(u), np.abs(v))
            assert np.array_equal(S, scale)


def check_alpha_zero_and_sign(orc):
    vals = si.uniform_f32(23, 0, 6 * 5, 0.0, 1.0)
    Apos = second_decode(si.f32_to_bf16_bits(vals), "bf16").reshape(6, 5)
    vals = si.uniform_f32(23, 1, 5 * 4, 0.0, 1.0)
    Bneg = -second_decode(si.f32_to_bf16_bits(vals), "bf16").reshape(5, 4)
    # alpha = 0 gives zeros, with or without the epilogue.
    for relu in (False, True):
        D = run(orc, Apos, Bneg, "bf16", 0.0, relu)
        assert np.all(D == 0.0)
    # A >= 0, B <= 0, alpha > 0: every product <= 0, ReLU clears all.
    D = run(orc, Apos, Bneg, "bf16", 1.25, True)
    assert np.all(D == 0.0) and not np.any(np.signbit(D))
    Dn = run(orc, Apos, Bneg, "bf16", 1.25, False)
    assert np.all(Dn < 0.0)
    # Negative alpha flips which entries survive: relu(alpha*s) = -alpha*|s| here.
    Dm = run(orc, Apos, Bneg, "bf16", -1.25, True)
    assert np.all(Dm > 0.0)
    assert np.array_equal(Dm, -Dn)


def exact_product(Alog, Blog, alpha, relu):
    """Exact rational D (as Fractions) for logical float inputs."""
    M, K = Alog.shape
    N = Blog.shape[1]
    out = [[None] * N for _ in range(M)]
    fa = Fraction(alpha)
    for i in range(M):
        for j in range(N):
            s = sum((Fraction(Alog[i, k]) * Fraction(Blog[k, j]) for k in range(K)), Fraction(0))
            y = fa * s
            if relu and y < 0:
                y = Fraction(0)
            out[i][j] = y
    return out


def check_bruteforce_exact(orc):
    """Tiny shapes on a dyadic grid (entries c/64, |c| <= 64): every double
    partial sum is exact, so the oracle must equal the exact rational result
    bit for bit, whatever the order."""
    for (M, N, K), seed in (((3, 4, 5), 31), ((5, 2, 9), 32), ((1, 7, 16), 33), ((8, 8, 3), 34)):
        ca = si.raw_u64(seed, 0, 0, M * K) % np.uint64(129)
        cb = si.raw_u64(seed, 1, 0, K * N) % np.uint64(129)
        Alog = (ca.astype(np.float64) - 64.0).reshape(M, K) / 64.0
        Blog = (cb.astype(np.float64) - 64.0).reshape(K, N) / 64.0
        # FP8 holds 2-3 fraction bits: a coarser grid (c/8, |c| <= 8).
        Alog8 = np.round(Alog * 8.0) / 8.0
        Blog8 = np.round(Blog * 8.0) / 8.0
        for dt in ("bf16", "fp16", "tf32", "e4m3", "e5m2"):
            if dt in ("e4m3", "e5m2"):
                for alpha, relu in ((1.0, False), (-1.5, True)):
                    D = run(orc, Alog8, Blog8, dt, alpha, relu)
                    E = exact_product(Alog8, Blog8, alpha, relu)
                    for i in range(M):
                        for j in range(N):
                            assert Fraction(D[i, j]) == E[i][j], (dt, M, N, K, i, j)
                continue
            for alpha, relu in ((1.0, False), (-1.5, True)):
                D = run(orc, Alog, Blog, dt, alpha, relu)
                E = exact_product(Alog, Blog, alpha, relu)
                for i in range(M):
                    for j in range(N):
                        assert Fraction(D[i, j]) == E[i][j], (dt, M, N, K, i, j)


def check_bruteforce_bound(orc):
    """Random bf16 in [-1, 1): the double sum is within K * 2^-53 * sum|ab|
    of the exact sum (the textbook bound for recursive summation)."""
    M, N, K = 4, 3, 12
    A = si.f32_to_bf16_bits(si.uniform_f32(41, 0, M * K, -1.0, 1.0)).reshape(M, K)
    B = si.f32_to_bf16_bits(si.uniform_f32(41, 1, N * K, -1.0, 1.0)).reshape(N, K)
    Alog = second_decode(A, "bf16")
    Blog = second_decode(B, "bf16").T
    D = orc.gemm(M, N, K, 1.0, A, K, B, K, "bf16", False)
    E = exact_product(Alog, Blog, 1.0, False)
    for i in range(M):
        for j in range(N):
            mag = sum(abs(Fraction(Alog[i, k]) * Fraction(Blog[k, j])) for k in range(K))
            assert abs(Fraction(D[i, j]) - E[i][j]) <= Fraction(K, 2 ** 53) * mag


def check_zero_padding_neutral(orc):
    """Embedding in a larger K with zero A columns / B rows changes nothing
    ('Matrix Multiplication', ragged sizes: zero padding is neutral)."""
    M, N, K, extra = 6, 5, 10, 7
    A = si.f32_to_bf16_bits(si.uniform_f32(51, 0, M * K, -1.0, 1.0)).reshape(M, K)
    B = si.f32_to_bf16_bits(si.uniform_f32(51, 1, N * K, -1.0, 1.0)).reshape(N, K)
    D0 = orc.gemm(M, N, K, 1.5, A, K, B, K, "bf16", True)
    Az = np.zeros((M, K + extra), np.uint16)
    Bz = np.zeros((N, K + extra), np.uint16)
    Az[:, :K] = A
    Bz[:, :K] = B
    D1 = orc.gemm(M, N, K + extra, 1.5, Az, K + extra, Bz, K + extra, "bf16", True)
    assert np.array_equal(D0, D1)


def check_strides_and_padding(orc):
    """lda > K and ldb > K with NaN padding: padding is never read, and the
    strided result equals the tight one."""
    w = si.Workload("t", 9, 7, 13, "bf16", 1.0, True, 52, "uniform", lda=21, ldb=16)
    A, B = si.make_operands(w)
    D = orc.gemm(9, 7, 13, 1.0, A, 21, B, 16, "bf16", True)
    assert not np.any(np.isnan(D))
    D2 = orc.gemm(9, 7, 13, 1.0, np.ascontiguousarray(A[:, :13]), 13,
                  np.ascontiguousarray(B[:, :13]), 13, "bf16", True)
    assert np.array_equal(D, D2)


def check_relu_special_values(orc):
    """Julia max semantics: NaN stays NaN, -0 becomes +0."""
    D = run(orc, [[1.0], [-1.0]], [[0.0, 1.0]], "bf16", 1.0, True)
    assert np.array_equal(D, [[0.0, 1.0], [0.0, 0.0]])
    assert not np.any(np.signbit(D))
    # A zero sum times a negative alpha is -0; the max with zero gives +0.
    D = run(orc, [[1.0], [2.0]], [[0.0, 0.0]], "bf16", -1.0, True)
    assert np.array_equal(D, np.zeros((2, 2))) and not np.any(np.signbit(D))
    Dn = run(orc, [[1.0], [2.0]], [[0.0, 0.0]], "bf16", -1.0, False)
    assert np.all(np.signbit(Dn))                 # without the epilogue -0 stays
    A = np.array([[np.nan, 1.0], [1.0, 1.0]], np.float32)
    Ab = (A.view(np.uint32) >> 16).astype(np.uint16)
    B = bf16_bits_exact(np.array([[1.0, 1.0], [-1.0, -1.0]]))  # storage row j = column j of B
    D = orc.gemm(2, 2, 2, 1.0, Ab, 2, B, 2, "bf16", True)
    assert np.isnan(D[0, 0]) and np.isnan(D[0, 1])
    assert D[1, 0] == 2.0 and D[1, 1] == 0.0


def check_entries_match_full(orc):
    w = si.Workload("e", 37, 29, 41, "fp16", 0.5, True, 61, "normal", scale=0.1, lda=45, ldb=48)
    A, B = si.make_operands(w)
    D, S = orc.gemm(37, 29, 41, 0.5, A, 45, B, 48, "fp16", True, with_scale=True)
    I = np.array([0, 36, 5, 17, 36, 0])
    J = np.array([0, 28, 11, 3, 0, 28])
    v, s = orc.gemm_entries(37, 29, 41, 0.5, A, 45, B, 48, "fp16", True, I, J)
    assert np.array_equal(v, D[I, J])
    assert np.array_equal(s, S[I, J])


def check_thread_independent(orc):
    w = si.Workload("t", 33, 17, 50, "bf16", 1.0, False, 62, "uniform")
    A, B = si.make_operands(w)
    D1 = orc.gemm(33, 17, 50, 1.0, A, 50, B, 50, "bf16", False, threads=1)
    D4 = orc.gemm(33, 17, 50, 1.0, A, 50, B, 50, "bf16", False, threads=4)
    assert np.array_equal(D1, D4)


def check_degenerate(orc):
    A = np.zeros((3, 1), np.uint16)
    B = np.zeros((4, 1), np.uint16)
    D = orc.gemm(3, 4, 0, 2.0, A, 1, B, 1, "bf16", True)
    assert D.shape == (3, 4) and np.all(D == 0.0)
    assert orc.gemm(0, 4, 5, 1.0, np.zeros(0, np.uint16), 5, np.zeros(20, np.uint16), 5,
                    "bf16", True).shape == (0, 4)
    assert orc.gemm(3, 0, 5, 1.0, np.zeros(15, np.uint16), 5, np.zeros(0, np.uint16), 5,
                    "bf16", True).shape == (3, 0)


def rne_reference(x: float, p: int, emin: int, emax: int) -> float:
    """Round to nearest even with exact rational arithmetic (a second
    formulation of the output rounding, independent of the oracle's)."""
    if math.isnan(x) or math.isinf(x) or x == 0.0:
        return x
    a = Fraction(abs(x))
    e = 0
    while a >= 2 ** (e + 1):
        e += 1
    while a < Fraction(2) ** e:
        e -= 1
    e = max(e, emin)
    quantum = Fraction(2) ** (e - (p - 1))
    q = a / quantum
    fl = q.numerator // q.denominator
    rem = q - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    out = fl * quantum
    if out > (2 - Fraction(2) ** (1 - p)) * Fraction(2) ** emax:
        return math.copysign(math.inf, x)
    return math.copysign(float(out), x)


def round_probe_values(seed=13, n=3000):
    vals = [1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11, 65504.0,
            65519.99, 65520.0, 65536.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14,
            (2 - 2 ** -8) * 2.0 ** 127, (2 - 2 ** -9) * 2.0 ** 127, 2.0 ** -133, 2.0 ** -134,
            3 * 2.0 ** -135, 1e-40, 3.4e38, -0.0, 0.0, math.inf, -math.inf, -1.5]
    u = si.raw_u64(seed, 0, 0, n)
    mant = (u >> np.uint64(11)).astype(np.float64) * 2.0 ** -53 + 1.0
    expo = (u % np.uint64(80)).astype(np.int64) - 40
    sign = np.where((u >> np.uint64(7)) & np.uint64(1), -1.0, 1.0)
    vals += list(sign * np.ldexp(mant, expo))
    return np.array(vals, dtype=np.float64)


def check_round_output(orc):
    """Output rounding ("convert on the way out") against numpy's own float32 /
    float16 conversions and an exact rational round-to-nearest-even."""
    x = round_probe_values()
    f32 = orc.round_output(x, "f32")
    with np.errstate(over="ignore"):
        assert np.array_equal(f32, x.astype(np.float32).astype(np.float64))
        f16 = orc.round_output(x, "fp16")
        want16 = x.astype(np.float16).astype(np.float64)
    assert np.array_equal(f16, want16)
    assert np.array_equal(np.signbit(f16), np.signbit(want16))
    bf = orc.round_output(x, "bf16")
    wantbf = np.array([rne_reference(float(v), 8, -126, 127) for v in x])
    assert np.array_equal(bf, wantbf)
    assert np.array_equal(np.signbit(bf), np.signbit(wantbf))
    # Hand-worked: bf16 keeps 8 significant bits; ties go to the even neighbour.
    hand = orc.round_output([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 255.5, 256.5, 257.0], "bf16")
    assert list(hand) == [1.0, 1.0 + 2 ** -6, 256.0, 256.0, 256.0]


def e5m2_by_fp16(codes: np.ndarray) -> np.ndarray:
    """E5M2 is the top byte of IEEE binary16 (same sign, 5-bit exponent with
    bias 15, top 2 fraction bits): decode through numpy's float16."""
    with np.errstate(invalid="ignore"):
        return (codes.astype(np.uint16) << 8).view(np.float16).astype(np.float64)


def e4m3_by_fp16(codes: np.ndarray) -> np.ndarray:
    """E4M3 re-encoded as binary16 bits (exponent bias 7 -> 15, 3 fraction
    bits -> the top of 10; subnormals shifted into normal fp16 numbers) and
    decoded by numpy: a second path to the same values."""
    out = np.empty(codes.shape, dtype=np.float64)
    for idx, c in enumerate(codes.astype(np.int64)):
        s, e, f = (c >> 7) & 1, (c >> 3) & 0xF, c & 7
        if e == 15 and f == 7:
            out[idx] = np.nan
            continue
        if e == 0:
            if f == 0:
                h = s << 15
            else:                      # f * 2^-9 = (f << shift) / 8 * 2^(-6 - shift)
                shift = 0
                while not (f & 8):
                    f <<= 1
                    shift += 1
                h = (s << 15) | ((-6 - shift + 15) << 10) | ((f & 7) << 7)
        else:
            h = (s << 15) | ((e - 7 + 15) << 10) | (f << 7)
        out[idx] = np.array([h], dtype=np.uint16).view(np.float16).astype(np.float64)[0]
    return out


def check_fp8_decode(orc):
    """All 256 E4M3 and E5M2 patterns against decodes through numpy's
    float16, the format's landmark values, sign symmetry and monotonicity."""
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    for dt, second in (("e5m2", e5m2_by_fp16), ("e4m3", e4m3_by_fp16)):
        got = orc.decode(codes, dt)
        want = second(codes)
        assert np.array_equal(np.isnan(got), np.isnan(want)), dt
        ok = ~np.isnan(want)
        assert np.array_equal(got[ok], want[ok]), dt
        assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok])), dt
        pos = got[:128]
        fin = pos[~np.isnan(pos) & ~np.isinf(pos)]
        assert np.all(np.diff(fin) > 0), dt                  # codes order the values
        assert np.array_equal(got[128:][ok[:128]], -got[:128][ok[:128]]), dt
    e4 = orc.decode(np.array([0x01, 0x08, 0x38, 0x7E, 0x7F, 0xFE], np.uint8), "e4m3")
    assert list(e4[[0, 1, 2, 3, 5]]) == [2.0 ** -9, 2.0 ** -6, 1.0, 448.0, -448.0]
    assert np.isnan(e4[4])
    e5 = orc.decode(np.array([0x01, 0x04, 0x3C, 0x7B, 0x7C, 0x7D], np.uint8), "e5m2")
    assert list(e5[:5]) == [2.0 ** -16, 2.0 ** -14, 1.0, 57344.0, math.inf] and np.isnan(e5[5])


# ---------------------------------------------------------------- block-scaled (MX) products

MX_GRID = np.arange(-8, 9) / 8.0     # exact in E4M3 and E5M2


# E2M1 values of codes 0..15 as the OCP format lists them (sign in bit 3).
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
              -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
FP4_GRID = np.array([-6, -4, -3, -2, -1.5, -1, -0.5, 0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)


def e2m1_codes_exact(vals) -> np.ndarray:
    v = np.asarray(vals, dtype=np.float64)
    out = np.zeros(v.shape, dtype=np.uint8)
    for idx, x in np.ndenumerate(v):
        hits = [c for c, t in enumerate(E2M1_TABLE)
                if t == x and math.copysign(1.0, t) == math.copysign(1.0, x)]
        assert hits, f"{x} not exact in e2m1"
        out[idx] = hits[0]
    return out


def mx_codes(vals, dtype):
    """Exact values (rows, K) -> storage rows: FP8 codes, or packed E2M1 with
    the row length rounded up to an even count (padding code +6)."""
    if dtype == "e2m1":
        v = np.asarray(vals, dtype=np.float64)
        rows, K = v.shape
        codes = np.full((rows, K + (K & 1)), 7, dtype=np.uint8)
        codes[:, :K] = e2m1_codes_exact(v)
        return np.ascontiguousarray((codes[:, 0::2] & 0xF) | ((codes[:, 1::2] & 0xF) << 4))
    return fp8_bits_exact(np.asarray(vals, dtype=np.float64), dtype)


def run_mx(orc, Alog, Blog, SAc, SBc, dtype, alpha, relu, pad_s=5, **kw):
    """Alog (M,K), Blog (K,N) exact FP8 values; SAc (M,KB), SBc (N,KB) scale
    codes.  Scale rows are stored with `pad_s` extra codes of padding (255,
    NaN) so a wrong block count or stride reads NaN into the result."""
    M, K = Alog.shape
    N = Blog.shape[1]
    KB = SAc.shape[1]
    A = mx_codes(Alog, dtype)
    B = np.ascontiguousarray(mx_codes(Blog.T, dtype))
    ld = K + (K & 1) if dtype == "e2m1" else K
    ldsa = ldsb = KB + pad_s
    SA = np.full((M, ldsa), 255, dtype=np.uint8)
    SB = np.full((N, ldsb), 255, dtype=np.uint8)
    SA[:, :KB] = SAc
    SB[:, :KB] = SBc
    return orc.gemm_mx(M, N, K, alpha, A, ld, SA, ldsa, B, ld, SB, ldsb, dtype, relu, **kw)


def check_mx_scale_decode(orc):
    """8-bit exponent scales: 2^(e-127) at the landmarks, exact doubling from
    code to code, NaN at 255."""
    got = orc.decode_scale(np.arange(256, dtype=np.uint16).astype(np.uint8))
    assert got[127] == 1.0 and got[128] == 2.0 and got[126] == 0.5
    assert got[0] == 2.0 ** -127 and got[254] == 2.0 ** 127
    assert np.all(got[1:255] == 2.0 * got[0:254])
    assert math.isnan(got[255])


def check_e2m1_decode(orc):
    """Every byte decodes to (low nibble, high nibble) per the E2M1 table."""
    got = orc.decode(np.arange(256, dtype=np.uint16).astype(np.uint8), "e2m1").reshape(256, 2)
    for b in range(256):
        for half, code in ((0, b & 0xF), (1, b >> 4)):
            want = E2M1_TABLE[code]
            assert got[b, half] == want and math.copysign(1.0, got[b, half]) == \
                math.copysign(1.0, want), (b, half)


def check_mx_bruteforce_exact(orc):
    """Tiny problems with ragged last blocks against exact rational
    arithmetic of the microscaling definition."""
    rng = np.random.default_rng(29)
    for (M, N, K) in ((3, 4, 70), (2, 5, 32), (4, 3, 97), (1, 1, 1)):
        KB = (K + 31) // 32
        SAc = rng.integers(121, 134, size=(M, KB)).astype(np.uint8)
        SBc = rng.integers(121, 134, size=(N, KB)).astype(np.uint8)
        for dt in ("e4m3", "e5m2", "e2m1"):
            grid = FP4_GRID if dt == "e2m1" else MX_GRID
            Alog = rng.choice(grid, size=(M, K))
            Blog = rng.choice(grid, size=(K, N))
            for alpha, relu in ((1.0, False), (-1.5, True)):
                D, S = run_mx(orc, Alog, Blog, SAc, SBc, dt, alpha, relu, with_scale=True)
                assert np.all(np.isfinite(D)) and np.all(np.isfinite(S)), (dt, M, N, K)
                for i in range(M):
                    for j in range(N):
                        s = Fraction(0)
                        t = Fraction(0)
                        for kb in range(KB):
                            x = Fraction(2) ** (int(SAc[i, kb]) - 127) * \
                                Fraction(2) ** (int(SBc[j, kb]) - 127)
                            ks = range(32 * kb, min(32 * kb + 32, K))
                            s += x * sum((Fraction(Alog[i, k]) * Fraction(Blog[k, j]) for k in ks),
                                         Fraction(0))
                            t += x * sum((abs(Fraction(Alog[i, k]) * Fraction(Blog[k, j])) for k in ks),
                                         Fraction(0))
                        y = Fraction(alpha) * s
                        if relu and y < 0:
                            y = Fraction(0)
                        assert Fraction(D[i, j]) == y, (dt, M, N, K, i, j)
                        assert Fraction(S[i, j]) == abs(Fraction(alpha)) * t


def check_mx_block_boundaries(orc):
    """A single one in row i at column k: D(i,j) = Xa(i, k // 32) * Xb(k // 32, j)
    exactly, at every block edge; pins the block size, the block offset and
    which scale row belongs to which operand row or column."""
    M, N, K = 2, 3, 100
    KB = 4
    SAc = np.array([[127 + kb + 4 * i for kb in range(KB)] for i in range(M)], dtype=np.uint8)
    SBc = np.array([[120 - 2 * kb - 9 * j for kb in range(KB)] for j in range(N)], dtype=np.uint8)
    Blog = np.ones((K, N))
    for dt in ("e4m3", "e2m1"):
        for k in (0, 1, 15, 16, 30, 31, 32, 33, 63, 64, 95, 96, 98, 99):
            Alog = np.zeros((M, K))
            Alog[0, k] = 1.0
            Alog[1, K - 1 - k] = -1.0
            Bk = Blog.copy()
            Bk[k, :] = 4.0       # the row meeting A's nonzero (pins E2M1 nibble order)
            Bk[K - 1 - k, :] = 2.0 if K - 1 - k != k else 4.0
            D = run_mx(orc, Alog, Bk, SAc, SBc, dt, 1.0, False)
            for j in range(N):
                kb0, kb1 = k // 32, (K - 1 - k) // 32
                want0 = Bk[k, j] * 2.0 ** (int(SAc[0, kb0]) - 127 + int(SBc[j, kb0]) - 127)
                want1 = -Bk[K - 1 - k, j] * 2.0 ** (int(SAc[1, kb1]) - 127 + int(SBc[j, kb1]) - 127)
                assert D[0, j] == want0 and D[1, j] == want1, (dt, k, j)


def check_mx_scale_invariances(orc):
    """One code step on every scale of row i of A doubles row i exactly; on
    every scale of column j of B doubles column j; nothing else moves."""
    rng = np.random.default_rng(31)
    M, N, K = 5, 6, 130
    KB = 5
    Alog = rng.choice(MX_GRID, size=(M, K))
    Blog = rng.choice(MX_GRID, size=(K, N))
    SAc = rng.integers(122, 132, size=(M, KB)).astype(np.uint8)
    SBc = rng.integers(122, 132, size=(N, KB)).astype(np.uint8)
    D = run_mx(orc, Alog, Blog, SAc, SBc, "e5m2", 0.75, False)
    SA2 = SAc.copy()
    SA2[3] += 1
    D2 = run_mx(orc, Alog, Blog, SA2, SBc, "e5m2", 0.75, False)
    assert np.array_equal(D2[3], 2 * D[3]) and np.array_equal(np.delete(D2, 3, 0), np.delete(D, 3, 0))
    SB2 = SBc.copy()
    SB2[4] -= 1
    D3 = run_mx(orc, Alog, Blog, SAc, SB2, "e5m2", 0.75, False)
    assert np.array_equal(D3[:, 4], D[:, 4] / 2)
    assert np.array_equal(np.delete(D3, 4, 1), np.delete(D, 4, 1))
    # All scales one: the unscaled product of the same codes.
    ones = run_mx(orc, Alog, Blog, np.full((M, KB), 127, np.uint8), np.full((N, KB), 127, np.uint8),
                  "e5m2", 0.75, False)
    A = mx_codes(Alog, "e5m2")
    B = np.ascontiguousarray(mx_codes(Blog.T, "e5m2"))
    assert np.array_equal(ones, orc.gemm(M, N, K, 0.75, A, K, B, K, "e5m2", False))


def check_mx_nan_scale(orc):
    """A NaN scale makes its whole row (or column) NaN, even where the block's
    elements are zero."""
    M, N, K = 3, 4, 64
    Alog = np.ones((M, K)) / 2
    Alog[1, 32:] = 0.0
    Blog = np.ones((K, N))
    SAc = np.full((M, 2), 127, np.uint8)
    SBc = np.full((N, 2), 127, np.uint8)
    SAc[1, 1] = 255
    SBc[2, 0] = 255
    D = run_mx(orc, Alog, Blog, SAc, SBc, "e4m3", 1.0, True)
    assert np.all(np.isnan(D[1])) and np.all(np.isnan(D[:, 2]))
    assert np.all(D[[0, 2]][:, [0, 1, 3]] == 32.0)


# ---------------------------------------------------------------- NVFP4 (16-element E4M3 scales)

def ue4m3_fraction(c: int) -> Fraction:
    """Unsigned E4M3 scale code as an exact rational, from the format: 4
    exponent bits (bias 7), 3 fraction bits, exponent 0 subnormal."""
    e, m = (c >> 3) & 0xF, c & 7
    if e == 0:
        return Fraction(m, 8) * Fraction(1, 64)
    return (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


def run_nv(orc, Alog, Blog, SAc, SBc, alpha, relu, pad_s=5, **kw):
    """Alog (M,K), Blog (K,N) exact E2M1 values; SAc (M,KB), SBc (N,KB)
    unsigned-E4M3 scale codes, KB = ceil(K/16).  Scale rows carry `pad_s`
    codes of NaN (0x7F) padding, so a wrong block count or stride shows."""
    M, K = Alog.shape
    N = Blog.shape[1]
    KB = SAc.shape[1]
    A = mx_codes(Alog, "e2m1")
    B = np.ascontiguousarray(mx_codes(Blog.T, "e2m1"))
    ld = K + (K & 1)
    ldsa = ldsb = KB + pad_s
    SA = np.full((M, ldsa), 0x7F, dtype=np.uint8)
    SB = np.full((N, ldsb), 0x7F, dtype=np.uint8)
    SA[:, :KB] = SAc
    SB[:, :KB] = SBc
    return orc.gemm_mx(M, N, K, alpha, A, ld, SA, ldsa, B, ld, SB, ldsb, "nvf4", relu, **kw)


def check_ue4m3_decode(orc):
    """The 128 unsigned E4M3 codes against E4M3 decoded through numpy's
    float16 (a second path), against exact rationals, and at the landmarks:
    1 at 0x38, 448 at 0x7E, 2^-9 at 0x01, 2^-6 at 0x08, NaN at 0x7F."""
    codes = np.arange(128, dtype=np.uint8)
    got = orc.decode_scale(codes, "ue4m3")
    want = e4m3_by_fp16(codes)
    assert np.array_equal(got[:127], want[:127]) and math.isnan(got[127])
    for c in range(127):
        assert Fraction(got[c]) == ue4m3_fraction(c), c
    assert (got[0x38], got[0x7E], got[0x01], got[0x08]) == (1.0, 448.0, 2.0 ** -9, 2.0 ** -6)
    assert np.all(np.diff(got[:127]) > 0)


def check_nvf4_bruteforce_exact(orc):
    """Tiny problems with ragged last blocks against exact rational
    arithmetic: 16-element blocks, each with its own pair of unsigned-E4M3
    scales (non-powers of two included)."""
    rng = np.random.default_rng(37)
    for (M, N, K) in ((3, 4, 70), (2, 5, 16), (4, 3, 33), (1, 1, 2), (2, 2, 48)):
        KB = (K + 15) // 16
        SAc = rng.integers(0x20, 0x50, size=(M, KB)).astype(np.uint8)
        SBc = rng.integers(0x20, 0x50, size=(N, KB)).astype(np.uint8)
        Alog = rng.choice(FP4_GRID, size=(M, K))
        Blog = rng.choice(FP4_GRID, size=(K, N))
        for alpha, relu in ((1.0, False), (-0.75, True)):
            D, S = run_nv(orc, Alog, Blog, SAc, SBc, alpha, relu, with_scale=True)
            for i in range(M):
                for j in range(N):
                    s = Fraction(0)
                    t = Fraction(0)
                    for kb in range(KB):
                        x = ue4m3_fraction(int(SAc[i, kb])) * ue4m3_fraction(int(SBc[j, kb]))
                        ks = range(16 * kb, min(16 * kb + 16, K))
                        s += x * sum((Fraction(Alog[i, k]) * Fraction(Blog[k, j]) for k in ks),
                                     Fraction(0))
                        t += x * sum((abs(Fraction(Alog[i, k]) * Fraction(Blog[k, j])) for k in ks),
                                     Fraction(0))
                    y = Fraction(alpha) * s
                    if relu and y < 0:
                        y = Fraction(0)
                    assert Fraction(D[i, j]) == y, (M, N, K, i, j)
                    assert Fraction(S[i, j]) == abs(Fraction(alpha)) * t


def check_nvf4_block_boundaries(orc):
    """A single nonzero in row i at column k: D(i,j) = b(k,j) * Xa(i, k // 16)
    * Xb(k // 16, j) exactly, at every block edge."""
    M, N, K = 2, 3, 70
    KB = 5
    SAc = np.array([[0x30 + 3 * kb + 5 * i for kb in range(KB)] for i in range(M)], dtype=np.uint8)
    SBc = np.array([[0x44 - 2 * kb - 7 * j for kb in range(KB)] for j in range(N)], dtype=np.uint8)
    for k in (0, 1, 15, 16, 17, 31, 32, 47, 48, 63, 64, 69):
        Alog = np.zeros((M, K))
        Alog[0, k] = 1.0
        Alog[1, K - 1 - k] = -1.5
        Bk = np.ones((K, N))
        Bk[k, :] = 4.0
        Bk[K - 1 - k, :] = 2.0 if K - 1 - k != k else 4.0
        D = run_nv(orc, Alog, Bk, SAc, SBc, 1.0, False)
        for j in range(N):
            kb0, kb1 = k // 16, (K - 1 - k) // 16
            want0 = Fraction(Bk[k, j]) * ue4m3_fraction(int(SAc[0, kb0])) * \
                ue4m3_fraction(int(SBc[j, kb0]))
            want1 = Fraction(-1.5) * Fraction(Bk[K - 1 - k, j]) * \
                ue4m3_fraction(int(SAc[1, kb1])) * ue4m3_fraction(int(SBc[j, kb1]))
            assert Fraction(D[0, j]) == want0 and Fraction(D[1, j]) == want1, (k, j)


def check_nvf4_unit_scales_and_codes(orc):
    """All scales 1 (code 0x38): the plain product of the E2M1 values (every
    partial sum of these quarter-integers is exact in double, so numpy's
    matmul gives it exactly) and the microscaling oracle with all scales 1;
    a NaN scale (0x7F) makes its row NaN; a code with the top bit set is
    refused."""
    rng = np.random.default_rng(41)
    M, N, K = 5, 4, 66
    Alog = rng.choice(FP4_GRID, size=(M, K))
    Blog = rng.choice(FP4_GRID, size=(K, N))
    D = run_nv(orc, Alog, Blog, np.full((M, 5), 0x38, np.uint8), np.full((N, 5), 0x38, np.uint8),
               1.25, False)
    assert np.array_equal(D, 1.25 * (Alog @ Blog))
    mx = run_mx(orc, Alog, Blog, np.full((M, 3), 127, np.uint8), np.full((N, 3), 127, np.uint8),
                "e2m1", 1.25, False)
    assert np.array_equal(D, mx)
    SAc = np.full((M, 5), 0x38, np.uint8)
    SAc[2, 4] = 0x7F
    Dn = run_nv(orc, Alog, Blog, SAc, np.full((N, 5), 0x38, np.uint8), 1.25, False)
    assert np.all(np.isnan(Dn[2])) and np.array_equal(np.delete(Dn, 2, 0), np.delete(D, 2, 0))
    SAc[2, 4] = 0x80
    try:
        run_nv(orc, Alog, Blog, SAc, np.full((N, 5), 0x38, np.uint8), 1.25, False)
    except ValueError:
        pass
    else:
        raise AssertionError("a scale code with the top bit set was accepted")


# ---------------------------------------------------------------- composed pointwise epilogues

def _epi_identity_case(vals):
    """A = I (M = K), B holding `vals` (K x N, exact BF16): s(i,j) = vals[i, j]."""
    M, N = vals.shape
    A = bf16_bits_exact(np.eye(M)).reshape(M, M)
    B = np.ascontiguousarray(bf16_bits_exact(vals.T))   # column j of B as row j
    return M, N, A, B


def run_epi(orc, vals, ops, alpha=1.0):
    M, N, A, B = _epi_identity_case(vals)
    return orc.gemm_epi(M, N, M, alpha, A, M, B, M, "bf16", ops)


def check_epi_pointwise_forms(orc):
    """Each op against its closed form at landmark points and its invariants."""
    ys = np.array([[-8.0, -2.0, -0.5, 0.0], [0.25, 1.0, 3.0, 10.0]])
    neg = -ys
    assert np.array_equal(run_epi(orc, ys, [("scale", -1.5, 0, None)]), -1.5 * ys)
    assert np.array_equal(run_epi(orc, ys, [("add", 0.75, 0, None)]), ys + 0.75)
    r = run_epi(orc, ys, [("relu", 0, 0, None)])
    assert np.array_equal(r, np.maximum(ys, 0.0)) and not np.any(np.signbit(r))
    assert np.array_equal(run_epi(orc, ys, [("leaky_relu", 0.125, 0, None)]),
                          np.where(ys > 0, ys, 0.125 * ys))
    assert np.array_equal(run_epi(orc, ys, [("clamp", -1.0, 2.0, None)]), np.clip(ys, -1.0, 2.0))
    sg, sgn = run_epi(orc, ys, [("sigmoid", 0, 0, None)]), run_epi(orc, neg, [("sigmoid", 0, 0, None)])
    assert sg[0, 3] == 0.5 and np.allclose(sg + sgn, 1.0, rtol=0, atol=1e-15)
    assert np.all((sg > 0) & (sg < 1)) and np.all(np.diff(sg[1]) > 0)
    si_ = run_epi(orc, ys, [("silu", 0, 0, None)])
    assert si_[0, 3] == 0.0 and np.allclose(si_, ys * sg, rtol=1e-15, atol=0)    # silu = y sigmoid(y)
    ge, gen = run_epi(orc, ys, [("gelu_tanh", 0, 0, None)]), run_epi(orc, neg, [("gelu_tanh", 0, 0, None)])
    assert ge[0, 3] == 0.0 and np.allclose(ge - gen, ys, rtol=0, atol=1e-14)      # odd tanh
    assert abs(ge[1, 3] - 10.0) < 1e-12 and abs(ge[0, 0]) < 1e-12                  # tails
    # Slope at 0 is 1/2; the cubic term bends it by 0.044715 * sqrt(2/pi) at small y.
    small = np.array([[1.0 / 1024, 1.0 / 256, 1.0 / 64, 1.0 / 16]])
    g = run_epi(orc, small, [("gelu_tanh", 0, 0, None)])
    k = math.sqrt(2.0 / math.pi)
    for y, gy in zip(small[0], g[0]):
        series = 0.5 * y + 0.5 * k * y * y + 0.5 * k * 0.044715 * y ** 4 - k ** 3 * y ** 4 / 6
        assert abs(gy - series) < 1e-6 * y ** 2, (y, gy, series)


def check_epi_composition_and_bias(orc):
    """Ops apply in list order after alpha; row biases follow i, column biases j."""
    rng = np.random.default_rng(37)
    vals = rng.integers(-8, 9, size=(5, 7)) / 8.0
    a1 = run_epi(orc, vals, [("scale", 2.0, 0, None), ("add", 1.0, 0, None)])
    a2 = run_epi(orc, vals, [("add", 1.0, 0, None), ("scale", 2.0, 0, None)])
    assert np.array_equal(a1, 2 * vals + 1) and np.array_equal(a2, 2 * vals + 2)
    al = run_epi(orc, vals, [("relu", 0, 0, None)], alpha=-1.0)
    assert np.array_equal(al, np.maximum(-vals, 0.0))
    br = np.arange(5, dtype=np.float32) * 0.5
    bc = np.arange(7, dtype=np.float32) * -0.25
    d = run_epi(orc, vals, [("bias_row", 0, 0, br), ("bias_col", 0, 0, bc)])
    assert np.array_equal(d, vals + br[:, None] + bc[None, :])
    assert np.array_equal(run_epi(orc, vals, []), vals)


def check_epi_nan(orc):
    """NaN passes the max-style ops (ReLU, leaky, clamp) as in the ReLU epilogue."""
    M, N = 3, 2
    A = bf16_bits_exact(np.eye(M)).reshape(M, M)
    B = np.ascontiguousarray(bf16_bits_exact(np.ones((N, M))))
    A[1, 1] = np.uint16(0x7FC0)
    for op in (("relu", 0, 0, None), ("leaky_relu", 0.5, 0, None), ("clamp", -1.0, 1.0, None)):
        d = orc.gemm_epi(M, N, M, 1.0, A, M, B, M, "bf16", [op])
        assert np.all(np.isnan(d[1])) and not np.any(np.isnan(d[[0, 2]])), op


def check_apply_epi_alone(orc):
    """The chain on given products (no GEMM): closed forms on a 5 x 7 array,
    row biases along i and column biases along j, the input left as it was."""
    rng = np.random.default_rng(41)
    y = rng.integers(-16, 17, size=(5, 7)) / 4.0
    keep = y.copy()
    br = (np.arange(5, dtype=np.float32) - 2) * 0.5
    bc = np.arange(7, dtype=np.float32) * 0.125
    d = orc.apply_epi(y, [("bias_row", 0, 0, br), ("clamp", -1.0, 1.5, None),
                          ("bias_col", 0, 0, bc), ("scale", 2.0, 0, None)])
    assert d.shape == (5, 7) and np.array_equal(y, keep)
    assert np.array_equal(d, 2.0 * (np.clip(y + br[:, None], -1.0, 1.5) + bc[None, :]))
    assert np.array_equal(orc.apply_epi(y, []), y)
    z = orc.apply_epi(np.zeros((3, 2)), [("add", 0.25, 0, None), ("sigmoid", 0, 0, None)])
    assert np.allclose(z, 1.0 / (1.0 + math.exp(-0.25)), rtol=1e-15, atol=0)


ALL_CHECKS = [
    check_decode_tables,
    check_tf32_narrowing,
    check_golden,
    check_identity,
    check_permutation,
    check_rank1,
    check_alpha_zero_and_sign,
    check_bruteforce_exact,
    check_bruteforce_bound,
    check_zero_padding_neutral,
    check_strides_and_padding,
    check_relu_special_values,
    check_entries_match_full,
    check_thread_independent,
    check_degenerate,
    check_round_output,
    check_fp8_decode,
    check_mx_scale_decode,
    check_e2m1_decode,
    check_mx_bruteforce_exact,
    check_mx_block_boundaries,
    check_mx_scale_invariances,
    check_mx_nan_scale,
    check_ue4m3_decode,
    check_nvf4_bruteforce_exact,
    check_nvf4_block_boundaries,
    check_nvf4_unit_scales_and_codes,
    check_epi_pointwise_forms,
    check_epi_composition_and_bias,
    check_epi_nan,
    check_apply_epi_alone,
]
