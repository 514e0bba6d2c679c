"""Seeded synthetic operands for the dense GEMM workloads.

This module is shared by the tests, the benchmark and the oracle's callers.
It only makes input bytes: it holds none of the GEMM's arithmetic (no
products, sums, scaling or epilogue).  Both the CUDA path and the oracle read
the very same buffers, so parity never depends on how a value was drawn.

Generator (defined here, not taken from any library so that it is the same
on every machine and every numpy version):

* ``splitmix64``: the 64-bit mixing function of Steele, Lea and Flood's
  SplitMix generator ("Fast splittable pseudorandom number generators",
  OOPSLA 2014): ``z = x + 0x9E3779B97F4A7C15; z = (z ^ z>>30) * 0xBF58476D1CE4E5B9;
  z = (z ^ z>>27) * 0x94D049BB133111EB; z ^ z>>31``.
* Element ``n`` of stream ``s`` under seed ``seed`` is
  ``splitmix64(key(seed, s) + n * 0x9E3779B97F4A7C15)`` with
  ``key(seed, s) = splitmix64(seed * 2**20 + s)``; it is counter-based, so any
  element can be regenerated on its own.
* A uniform in [0, 1) takes the top 24 bits: ``(x >> 40) * 2**-24`` (exact in
  float32).  ``[lo, hi)`` maps by ``lo + (hi - lo) * u`` in float64 then
  rounds to float32 (exact for [-1, 1) and [0, 1)).
* A standard normal uses Box-Muller on two uniforms of one element:
  ``u1`` from counter ``2n``, ``u2`` from ``2n + 1``,
  ``sqrt(-2 ln(1 - u1)) * cos(2 pi u2)`` in float64, then float32.

Operands are "rounded to BF16/FP16" from float32 by IEEE round to nearest,
ties to even; FP8 (E4M3/E5M2) operands take the nearest code (ties to the
even code, saturating at the largest finite value).  TF32 workloads keep float32 storage; the narrowing is the
method's own step and happens inside the GEMM, not here.

Storage follows the GEMM's conventions (Walk through GEMM, section 2 "Bind
runtime global arrays"): A is logically (M, K) and K-contiguous with leading
stride ``lda`` (numpy array of shape (M, lda)); B is logically (K, N) and
K-contiguous with ``ldb`` (numpy shape (N, ldb)); D is (M, N) M-contiguous
with ``ldc`` (numpy shape (N, ldc)).  Stride padding is filled with a NaN
sentinel so that a kernel reading it shows up at once.
"""

from __future__ import annotations

import dataclasses
import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# NaN sentinels written into stride padding (quiet NaNs of each storage type).
PAD_BF16 = 0x7FC1
PAD_FP16 = 0x7E01
PAD_F32_BITS = 0x7FC00001

STREAM_A = 0
STREAM_B = 1
STREAM_SA = 2   # block scales of A (microscaling workloads)
STREAM_SB = 3   # block scales of B


def splitmix64(x: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array (wrapping arithmetic)."""
    with np.errstate(over="ignore"):
        z = (x + _GAMMA).astype(np.uint64)
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _stream_key(seed: int, stream: int) -> np.uint64:
    base = np.array([(int(seed) << 20) + int(stream)], dtype=np.uint64)
    return splitmix64(base)[0]


def raw_u64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Counter-based 64-bit draws ``start .. start+count-1`` of one stream."""
    key = _stream_key(seed, stream)
    n = np.arange(start, start + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return splitmix64(key + n * _GAMMA)


def uniform01(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Uniform float64 values on the 2**-24 grid of [0, 1)."""
    x = raw_u64(seed, stream, start, count)
    return (x >> np.uint64(40)).astype(np.float64) * (2.0 ** -24)


CHUNK = 1 << 20  # elements generated per pass (keeps temporaries in cache)


def uniform_f32(seed: int, stream: int, count: int, lo: float, hi: float) -> np.ndarray:
    out = np.empty(count, dtype=np.float32)
    for s0 in range(0, count, CHUNK):
        n = min(CHUNK, count - s0)
        u = uniform01(seed, stream, s0, n)
        out[s0:s0 + n] = lo + (hi - lo) * u
    return out


def normal_f32(seed: int, stream: int, count: int, scale: float = 1.0) -> np.ndarray:
    out = np.empty(count, dtype=np.float32)
    for s0 in range(0, count, CHUNK):
        n = min(CHUNK, count - s0)
        u = uniform01(seed, stream, 2 * s0, 2 * n)
        u1 = u[0::2]
        u2 = u[1::2]
        z = np.sqrt(-2.0 * np.log1p(-u1)) * np.cos((2.0 * np.pi) * u2)
        out[s0:s0 + n] = z * scale
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """IEEE round-to-nearest-even float32 -> bfloat16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).reshape(-1)
    out = np.empty(u.shape, dtype=np.uint16)
    for s0 in range(0, u.size, CHUNK):
        c = u[s0:s0 + CHUNK]
        with np.errstate(over="ignore"):
            r = (c + np.uint32(0x7FFF) + ((c >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
        nan = (c & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
        if nan.any():
            r = np.where(nan, (c >> np.uint32(16)) | np.uint32(0x40), r)
        out[s0:s0 + CHUNK] = r
    return out.reshape(np.shape(x))


def f32_to_fp16_bits(x: np.ndarray) -> np.ndarray:
    """IEEE round-to-nearest-even float32 -> binary16 bit patterns."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


# (exponent bias, fraction bits, largest finite value) of the two OCP FP8 formats.
_FP8 = {"e4m3": (7, 3, 448.0), "e5m2": (15, 2, 57344.0)}


def f32_to_fp8_bits(x: np.ndarray, fmt: str) -> np.ndarray:
    """Round float32 values to the nearest E4M3 / E5M2 code (ties to the even
    code), saturating at the largest finite value; NaN -> code 0x7F (NaN in
    both formats)."""
    bias, mbits, top = _FP8[fmt]
    x64 = np.asarray(x, dtype=np.float64).reshape(-1)
    a = np.abs(x64)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    emin = 1 - bias
    # Quantum of the binade holding |x| (the subnormal quantum below 2^emin).
    _, ex = np.frexp(a)
    e = np.maximum(ex - 1, emin)
    q = np.ldexp(1.0, e - mbits)
    r = np.minimum(np.round(a / q) * q, top)       # np.round: ties to even
    # Encode: subnormal codes count quanta of 2^(emin - mbits); normal codes
    # hold (biased exponent, fraction).
    _, er = np.frexp(r)
    er = er - 1
    sub = r < 2.0 ** emin
    code_sub = np.round(r / 2.0 ** (emin - mbits))
    code_norm = ((er + bias) << mbits) + (np.ldexp(r, mbits - er) - (1 << mbits))
    code = np.where(sub, code_sub, code_norm).astype(np.uint8)
    code = np.where(np.signbit(x64), code | 0x80, code).astype(np.uint8)
    code[nan] = 0x7F
    return code.reshape(np.shape(x))


DTYPES = ("bf16", "fp16", "tf32", "e4m3", "e5m2")


# E2M1 (FP4): magnitudes of codes 0..7; no infinities or NaN.
E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
PAD_E2M1 = 0x7  # +6: stride padding of packed FP4 rows (never read)


def f32_to_e2m1_codes(x: np.ndarray) -> np.ndarray:
    """Round to the nearest E2M1 code (ties to the even code), saturating at
    6; 4-bit codes in uint8 (sign in bit 3).  NaN is not representable and
    maps to +6."""
    x64 = np.asarray(x, dtype=np.float64).reshape(-1)
    a = np.abs(np.where(np.isnan(x64), 6.0, x64))
    hi = np.clip(np.searchsorted(E2M1_VALUES, a), 1, 7)
    lo = hi - 1
    dlo, dhi = a - E2M1_VALUES[lo], E2M1_VALUES[hi] - a
    pick = np.where((dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0)), hi, lo)
    pick = np.where(a >= 6.0, 7, pick).astype(np.uint8)
    sign = np.signbit(x64) & ~np.isnan(x64)
    return np.where(sign, pick | 0x8, pick).astype(np.uint8).reshape(np.shape(x))


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """(..., 2n) 4-bit codes -> (..., n) bytes, element 2t in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def element_bytes(dtype: str) -> float:
    return {"bf16": 2, "fp16": 2, "tf32": 4, "e4m3": 1, "e5m2": 1, "e2m1": 0.5,
            "nvf4": 0.5}[dtype]


def storage_numpy_dtype(dtype: str):
    return {"bf16": np.uint16, "fp16": np.uint16, "tf32": np.float32, "e4m3": np.uint8,
            "e5m2": np.uint8, "e2m1": np.uint8, "nvf4": np.uint8}[dtype]


def scale_block(dtype: str) -> int:
    """K elements per block scale: 32 (8-bit exponent scales), or 16 for
    "nvf4" (packed E2M1 with unsigned-E4M3 scales)."""
    return 16 if dtype == "nvf4" else 32


@dataclasses.dataclass(frozen=True)
class Workload:
    """One GEMM problem: shapes, strides, operand type, scalars and the
    distribution its entries are drawn from."""

    name: str
    M: int
    N: int
    K: int
    dtype: str
    alpha: float
    relu: bool
    seed: int
    dist: str  # "uniform" or "normal"
    lo: float = -1.0
    hi: float = 1.0
    scale: float = 1.0
    lda: int | None = None
    ldb: int | None = None
    ldc: int | None = None
    block_scaled: bool = False  # one scale per 32 K (8-bit exponent) or per 16 K ("nvf4")

    @property
    def strides(self):
        return (self.lda or max(self.K, 1), self.ldb or max(self.K, 1), self.ldc or max(self.M, 1))

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    @property
    def algorithmic_bytes(self) -> float:
        e = element_bytes(self.dtype)
        kb = -(-self.K // scale_block(self.dtype))
        scales = (self.M + self.N) * kb if self.block_scaled else 0
        return float((self.M * self.K + self.K * self.N) * e + scales + 4 * self.M * self.N)


# The problems the pages and their configurations fix.
WORKLOADS = {
    # Walk through GEMM example run 65 x 97 x 73 (bounded edge tiles, TMA-illegal strides).
    "c1_bf16_65x97x73": Workload("c1_bf16_65x97x73", 65, 97, 73, "bf16", 1.5, True, 0, "uniform", -1.0, 1.0),
    # cuTile tutorial step-3/4 shape, FP32 operands narrowed to TF32.
    "c2_tf32_256x128x512": Workload("c2_tf32_256x128x512", 256, 128, 512, "tf32", 1.0, False, 1, "uniform", 0.0, 1.0),
    "c3_fp16_4096": Workload("c3_fp16_4096", 4096, 4096, 4096, "fp16", 0.5, True, 2, "normal", scale=0.1),
    "c4_bf16_8192": Workload("c4_bf16_8192", 8192, 8192, 8192, "bf16", 1.0, True, 3, "normal"),
    "c5a_bf16_16384x64x4096": Workload("c5a_bf16_16384x64x4096", 16384, 64, 4096, "bf16", 1.0, True, 4, "uniform",
                                       lda=4104, ldb=4104, ldc=16392),
    "c5b_bf16_64x16384x4096": Workload("c5b_bf16_64x16384x4096", 64, 16384, 4096, "bf16", 1.0, True, 4, "uniform",
                                       lda=4104, ldb=4104, ldc=72),
    "c5c_bf16_8191x4097x1000": Workload("c5c_bf16_8191x4097x1000", 8191, 4097, 1000, "bf16", 1.0, True, 4, "uniform",
                                        lda=1008, ldb=1008, ldc=8199),
    # 8-bit float operands at the headline size ("Matrix Multiplication",
    # "Where to go from here": FP8 matmuls), N(0,1) entries rounded to the type.
    "f8_e4m3_8192": Workload("f8_e4m3_8192", 8192, 8192, 8192, "e4m3", 1.0, True, 6, "normal"),
    "f8_e5m2_8192": Workload("f8_e5m2_8192", 8192, 8192, 8192, "e5m2", 1.0, True, 7, "normal"),
    # Block-scaled (microscaling) E4M3 at the headline size: N(0,1) entries
    # rounded to E4M3, one scale 2^e, e in [-7, 7], per 32 K elements.
    "mx_e4m3_8192": Workload("mx_e4m3_8192", 8192, 8192, 8192, "e4m3", 1.0, True, 8, "normal",
                             block_scaled=True),
    # The same with packed E2M1 (FP4) operands: N(0,1) rounded to E2M1.
    "mx_e2m1_8192": Workload("mx_e2m1_8192", 8192, 8192, 8192, "e2m1", 1.0, True, 9, "normal",
                             block_scaled=True),
    # NVFP4: the same packed E2M1 operands, one unsigned-E4M3 scale per 16 K.
    "nvf4_8192": Workload("nvf4_8192", 8192, 8192, 8192, "nvf4", 1.0, True, 10, "normal",
                          block_scaled=True),
}


def _draw(w: Workload, stream: int, count: int) -> np.ndarray:
    if w.dist == "uniform":
        return uniform_f32(w.seed, stream, count, w.lo, w.hi)
    if w.dist == "normal":
        return normal_f32(w.seed, stream, count, w.scale)
    raise ValueError(w.dist)


def _to_storage(x32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return f32_to_bf16_bits(x32)
    if dtype == "fp16":
        return f32_to_fp16_bits(x32)
    if dtype in ("e4m3", "e5m2"):
        flat = np.asarray(x32).reshape(-1)
        out = np.empty(flat.size, dtype=np.uint8)
        for s0 in range(0, flat.size, CHUNK):
            out[s0: s0 + CHUNK] = f32_to_fp8_bits(flat[s0: s0 + CHUNK], dtype)
        return out.reshape(np.shape(x32))
    if dtype == "tf32":
        return np.ascontiguousarray(x32, dtype=np.float32)
    raise ValueError(dtype)


def pad_value(dtype: str):
    if dtype == "bf16":
        return np.uint16(PAD_BF16)
    if dtype == "fp16":
        return np.uint16(PAD_FP16)
    if dtype in ("e4m3", "e5m2"):
        return np.uint8(0x7F)      # NaN in both FP8 formats
    return np.array([PAD_F32_BITS], dtype=np.uint32).view(np.float32)[0]


def make_operands(w: Workload):
    """Return (A, B) storage arrays for workload ``w``.

    A has shape (M, lda): row i holds A[i, 0:K] then NaN padding.
    B has shape (N, ldb): row j holds B[0:K, j] then NaN padding.
    (E2M1: packed, shapes (M, lda/2) and (N, ldb/2) bytes; padding +6.)
    A's logical entries use stream 0 in row-major (i, k) order, B's use
    stream 1 in (j, k) order.
    """
    lda, ldb, _ = w.strides
    if w.dtype in ("e2m1", "nvf4"):
        # Packed FP4: rows of lda / 2 bytes (lda even), padding code +6.
        assert lda % 2 == 0 and ldb % 2 == 0, "E2M1 rows must hold an even number of elements"
        out = []
        for rows, ld, stream in ((w.M, lda, STREAM_A), (w.N, ldb, STREAM_B)):
            codes = np.full((rows, ld), PAD_E2M1, dtype=np.uint8)
            if rows * w.K:
                flat = _draw(w, stream, rows * w.K)
                q = np.empty(flat.size, dtype=np.uint8)
                for s0 in range(0, flat.size, CHUNK):
                    q[s0: s0 + CHUNK] = f32_to_e2m1_codes(flat[s0: s0 + CHUNK])
                codes[:, : w.K] = q.reshape(rows, w.K)
            out.append(pack_e2m1(codes))
        return out[0], out[1]
    A = np.full((w.M, lda), pad_value(w.dtype), dtype=storage_numpy_dtype(w.dtype))
    B = np.full((w.N, ldb), pad_value(w.dtype), dtype=storage_numpy_dtype(w.dtype))
    if w.M * w.K:
        A[:, : w.K] = _to_storage(_draw(w, STREAM_A, w.M * w.K), w.dtype).reshape(w.M, w.K)
    if w.N * w.K:
        B[:, : w.K] = _to_storage(_draw(w, STREAM_B, w.N * w.K), w.dtype).reshape(w.N, w.K)
    return A, B


def make_output(w: Workload, fill_bits: int = 0x7FC00002) -> np.ndarray:
    """D storage of shape (N, ldc) filled with a float32 NaN sentinel, so the
    rows i >= M of each column (stride padding) can be checked untouched."""
    _, _, ldc = w.strides
    return np.full((w.N, ldc), fill_bits, dtype=np.uint32).view(np.float32)


def scale_codes(seed: int, stream: int, rows: int, kblocks: int, lo: int, hi: int) -> np.ndarray:
    """(rows, kblocks) uint8 scale exponent codes drawn uniformly from
    [lo, hi], row-major from draw 0 of the stream."""
    n = rows * kblocks
    out = np.empty(n, dtype=np.uint8)
    span = np.uint64(hi - lo + 1)
    for s0 in range(0, n, CHUNK):
        c = min(CHUNK, n - s0)
        out[s0: s0 + c] = (raw_u64(seed, stream, s0, c) % span + np.uint64(lo)).astype(np.uint8)
    return out.reshape(rows, kblocks)


MX_BENCH_SCALES = (120, 134)   # codes of the benchmark's block scales: 2^-7 .. 2^7
# Unsigned-E4M3 scale codes of "nvf4" workloads: 0x28 .. 0x48 = 0.25 .. 4,
# every mantissa in between (0x7F would be NaN).
NV_SCALES = (0x28, 0x48)


def bench_scales(dtype: str):
    return NV_SCALES if dtype == "nvf4" else MX_BENCH_SCALES


def make_mx_scales(w: Workload, lo: int | None = None, hi: int | None = None):
    """Row-major block scales (one per scale_block(w.dtype) K elements) for
    A's M rows and B's N columns of workload ``w``: codes drawn uniformly from
    [lo, hi] (default: bench_scales of the type)."""
    dlo, dhi = bench_scales(w.dtype)
    lo = dlo if lo is None else lo
    hi = dhi if hi is None else hi
    kb = -(-w.K // scale_block(w.dtype))
    return (scale_codes(w.seed, STREAM_SA, w.M, kb, lo, hi),
            scale_codes(w.seed, STREAM_SB, w.N, kb, lo, hi))


def with_shape(w: Workload, **kw) -> Workload:
    return dataclasses.replace(w, **kw)
