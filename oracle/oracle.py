"""ctypes binding and build step for ``oracle_gemm.c``.

TEST INFRASTRUCTURE ONLY (see the package docstring).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle_gemm.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD_DIR, "liboracle_gemm.so")

_DTYPE_CODE = {"bf16": 0, "fp16": 1, "tf32": 2, "e4m3": 3, "e5m2": 4, "e2m1": 5, "nvf4": 5}
_STORAGE = {"bf16": np.uint16, "fp16": np.uint16, "tf32": np.float32, "e4m3": np.uint8,
            "e5m2": np.uint8, "e2m1": np.uint8, "nvf4": np.uint8}
# Elements per storage unit (E2M1: two per byte, low nibble first; "nvf4" is
# E2M1 storage with 16-element unsigned-E4M3 block scales).
_PER_UNIT = {"e2m1": 2, "nvf4": 2}
# K elements per block scale.
SCALE_BLOCK = {"e4m3": 32, "e5m2": 32, "e2m1": 32, "nvf4": 16}
_OUT_CODE = {"f32": 0, "bf16": 1, "fp16": 2}
EPI_KINDS = {"scale": 0, "add": 1, "relu": 2, "leaky_relu": 3, "clamp": 4, "sigmoid": 5,
             "silu": 6, "gelu_tanh": 7, "bias_row": 8, "bias_col": 9}
GCC_FLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread"]

_lock = threading.Lock()
_default = None


def library_path() -> str:
    return _LIB


def compile_source(src: str, out: str) -> str:
    """gcc-compile one oracle source file into a shared library."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".tmp.%d" % os.getpid()
    subprocess.run(["gcc", *GCC_FLAGS, src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no GPU needed).  Returns the .so path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_source(SOURCE, _LIB)
    return _LIB


def _check_storage(x, dtype: str, name: str) -> np.ndarray:
    x = np.asarray(x)
    want = _STORAGE[dtype]
    if x.dtype != want:
        raise TypeError(f"{name}: {dtype} storage must be {np.dtype(want).name}, got {x.dtype}")
    return np.ascontiguousarray(x)


class Oracle:
    """One loaded copy of the oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, dbl, vp, ip = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
        lib.orc_gemm.argtypes = [i64, i64, i64, dbl, vp, i64, vp, i64, ip, ip, vp, i64, vp, ip]
        lib.orc_gemm.restype = ip
        lib.orc_gemm_entries.argtypes = [i64, i64, i64, dbl, vp, i64, vp, i64, ip, ip, vp, vp, i64,
                                         vp, vp, ip]
        lib.orc_gemm_entries.restype = ip
        lib.orc_decode_array.argtypes = [vp, i64, ip, vp]
        lib.orc_decode_array.restype = None
        lib.orc_round_output.argtypes = [vp, i64, ip]
        lib.orc_round_output.restype = None
        lib.orc_gemm_mx.argtypes = [i64, i64, i64, dbl, vp, i64, vp, i64, vp, i64, vp, i64, ip, ip,
                                    vp, i64, vp, ip]
        lib.orc_gemm_mx.restype = ip
        lib.orc_decode_e8m0_array.argtypes = [vp, i64, vp]
        lib.orc_decode_e8m0_array.restype = None
        lib.orc_gemm_nvf4.argtypes = [i64, i64, i64, dbl, vp, i64, vp, i64, vp, i64, vp, i64, ip,
                                      vp, i64, vp, ip]
        lib.orc_gemm_nvf4.restype = ip
        lib.orc_decode_ue4m3_array.argtypes = [vp, i64, vp]
        lib.orc_decode_ue4m3_array.restype = None
        lib.orc_gemm_epi.argtypes = [i64, i64, i64, dbl, vp, i64, vp, i64, ip, vp, vp, vp, vp, ip,
                                     vp, i64, vp, ip]
        lib.orc_gemm_epi.restype = ip
        lib.orc_apply_epi.argtypes = [i64, i64, vp, vp, vp, vp, ip, vp, i64]
        lib.orc_apply_epi.restype = ip
        lib.orc_num_host_threads.argtypes = []
        lib.orc_num_host_threads.restype = ip
        self.lib = lib
        self.path = path

    def host_threads(self) -> int:
        return int(self.lib.orc_num_host_threads())

    def gemm(self, M, N, K, alpha, A, lda, B, ldb, dtype, relu, with_scale=False, threads=0):
        """Full D_ref as a (M, N) float64 array (and |alpha|*sum|a||b| if asked).

        ``A``/``B`` are flat or 2-D storage arrays: a(i,k) = A.flat[i*lda + k],
        b(k,j) = B.flat[k + j*ldb].  bf16/fp16 storage is uint16 bit patterns,
        e4m3/e5m2 storage uint8 bit patterns, tf32 storage float32.
        """
        A = _check_storage(A, dtype, "A")
        B = _check_storage(B, dtype, "B")
        if M and K and A.size < (M - 1) * lda + K:
            raise ValueError("A too small for (M, K, lda)")
        if N and K and B.size < (N - 1) * ldb + K:
            raise ValueError("B too small for (K, N, ldb)")
        Dt = np.zeros((max(N, 0), max(M, 0)), dtype=np.float64)  # column-major (M, N)
        St = np.zeros_like(Dt) if with_scale else None
        rc = self.lib.orc_gemm(M, N, K, float(alpha), A.ctypes.data, lda, B.ctypes.data, ldb,
                               _DTYPE_CODE[dtype], int(bool(relu)), Dt.ctypes.data, max(M, 1),
                               St.ctypes.data if St is not None else None, int(threads))
        if rc != 0:
            raise ValueError(f"orc_gemm failed with {rc}")
        return (Dt.T, St.T) if with_scale else Dt.T

    def gemm_mx(self, M, N, K, alpha, A, lda, SA, ldsa, B, ldb, SB, ldsb, dtype, relu,
                with_scale=False, threads=0):
        """Block-scaled D_ref (M, N) float64: FP8 operands as in ``gemm``, and
        one 8-bit exponent scale per 32 k, Xa(i,kb) = SA.flat[i*ldsa + kb],
        Xb(kb,j) = SB.flat[j*ldsb + kb] (uint8 codes).  For e2m1, A and B are
        packed bytes and lda, ldb count elements (even).  dtype "nvf4": packed
        E2M1 with one unsigned-E4M3 scale per 16 k (orc_gemm_nvf4)."""
        A = _check_storage(A, dtype, "A")
        B = _check_storage(B, dtype, "B")
        per = _PER_UNIT.get(dtype, 1)
        SA = np.ascontiguousarray(SA, dtype=np.uint8)
        SB = np.ascontiguousarray(SB, dtype=np.uint8)
        blk = SCALE_BLOCK[dtype]
        kb = (K + blk - 1) // blk
        if M and K and A.size * per < (M - 1) * lda + K:
            raise ValueError("A too small for (M, K, lda)")
        if N and K and B.size * per < (N - 1) * ldb + K:
            raise ValueError("B too small for (K, N, ldb)")
        if M and kb and SA.size < (M - 1) * ldsa + kb:
            raise ValueError("SA too small")
        if N and kb and SB.size < (N - 1) * ldsb + kb:
            raise ValueError("SB too small")
        Dt = np.zeros((max(N, 0), max(M, 0)), dtype=np.float64)
        St = np.zeros_like(Dt) if with_scale else None
        sp = St.ctypes.data if St is not None else None
        if dtype == "nvf4":
            rc = self.lib.orc_gemm_nvf4(M, N, K, float(alpha), A.ctypes.data, lda, SA.ctypes.data,
                                        ldsa, B.ctypes.data, ldb, SB.ctypes.data, ldsb,
                                        int(bool(relu)), Dt.ctypes.data, max(M, 1), sp,
                                        int(threads))
        else:
            rc = self.lib.orc_gemm_mx(M, N, K, float(alpha), A.ctypes.data, lda, SA.ctypes.data,
                                      ldsa, B.ctypes.data, ldb, SB.ctypes.data, ldsb,
                                      _DTYPE_CODE[dtype], int(bool(relu)), Dt.ctypes.data,
                                      max(M, 1), sp, int(threads))
        if rc != 0:
            raise ValueError(f"block-scaled oracle failed with {rc}")
        return (Dt.T, St.T) if with_scale else Dt.T

    def decode_scale(self, codes, fmt: str = "e8m0") -> np.ndarray:
        """The oracle's decode of scale codes to float64: 8-bit exponents
        ("e8m0", the microscaling kinds) or unsigned E4M3 ("ue4m3", nvf4)."""
        x = np.ascontiguousarray(codes, dtype=np.uint8)
        out = np.zeros(x.shape, dtype=np.float64)
        fn = {"e8m0": self.lib.orc_decode_e8m0_array,
              "ue4m3": self.lib.orc_decode_ue4m3_array}[fmt]
        fn(x.ctypes.data, x.size, out.ctypes.data)
        return out

    @staticmethod
    def _ops(ops):
        n = len(ops)
        kinds = np.array([EPI_KINDS[o[0]] for o in ops] or [0], dtype=np.int32)
        av = np.array([float(o[1]) for o in ops] or [0.0], dtype=np.float64)
        bv = np.array([float(o[2]) for o in ops] or [0.0], dtype=np.float64)
        keep = [np.ascontiguousarray(o[3], dtype=np.float32) if o[3] is not None else None
                for o in ops]
        ptrs = (ctypes.c_void_p * max(n, 1))(*[k.ctypes.data if k is not None else None
                                               for k in keep] or [None])
        return n, kinds, av, bv, keep, ptrs

    def apply_epi(self, y, ops) -> np.ndarray:
        """The op chain of ``gemm_epi`` alone, on an (M, N) array of products
        y = alpha * s; returns a new float64 array."""
        Dt = np.array(np.asarray(y, dtype=np.float64).T, dtype=np.float64, order="C", copy=True)
        N, M = Dt.shape
        n, kinds, av, bv, keep, ptrs = self._ops(ops)
        rc = self.lib.orc_apply_epi(M, N, kinds.ctypes.data, av.ctypes.data, bv.ctypes.data,
                                    ctypes.cast(ptrs, ctypes.c_void_p), n, Dt.ctypes.data,
                                    max(M, 1))
        if rc != 0:
            raise ValueError(f"orc_apply_epi failed with {rc}")
        return Dt.T

    def gemm_epi(self, M, N, K, alpha, A, lda, B, ldb, dtype, ops, with_scale=False, threads=0):
        """D_ref with a composed pointwise epilogue: y = alpha * s, then each
        op of ``ops`` in order; an op is (kind, a, b, bias) with kind a name
        of EPI_KINDS and bias a float32 array (or None)."""
        A = _check_storage(A, dtype, "A")
        B = _check_storage(B, dtype, "B")
        n, kinds, av, bv, keep, ptrs = self._ops(ops)
        Dt = np.zeros((max(N, 0), max(M, 0)), dtype=np.float64)
        St = np.zeros_like(Dt) if with_scale else None
        rc = self.lib.orc_gemm_epi(M, N, K, float(alpha), A.ctypes.data, lda, B.ctypes.data, ldb,
                                   _DTYPE_CODE[dtype], kinds.ctypes.data, av.ctypes.data,
                                   bv.ctypes.data, ctypes.cast(ptrs, ctypes.c_void_p), n,
                                   Dt.ctypes.data, max(M, 1),
                                   St.ctypes.data if St is not None else None, int(threads))
        if rc != 0:
            raise ValueError(f"orc_gemm_epi failed with {rc}")
        return (Dt.T, St.T) if with_scale else Dt.T

    def gemm_entries(self, M, N, K, alpha, A, lda, B, ldb, dtype, relu, I, J, threads=0):
        """D_ref and |alpha|*sum|a||b| at coordinates (I[q], J[q])."""
        A = _check_storage(A, dtype, "A")
        B = _check_storage(B, dtype, "B")
        I = np.ascontiguousarray(I, dtype=np.int64)
        J = np.ascontiguousarray(J, dtype=np.int64)
        if I.shape != J.shape:
            raise ValueError("I and J differ in shape")
        out = np.zeros(I.shape, dtype=np.float64)
        scale = np.zeros(I.shape, dtype=np.float64)
        rc = self.lib.orc_gemm_entries(M, N, K, float(alpha), A.ctypes.data, lda, B.ctypes.data, ldb,
                                       _DTYPE_CODE[dtype], int(bool(relu)), I.ctypes.data,
                                       J.ctypes.data, I.size, out.ctypes.data, scale.ctypes.data,
                                       int(threads))
        if rc != 0:
            raise ValueError(f"orc_gemm_entries failed with {rc}")
        return out, scale

    def round_output(self, y, out_dtype: str) -> np.ndarray:
        """The output step: round float64 values to fp32 / bf16 / fp16 (RNE)."""
        arr = np.array(y, dtype=np.float64, copy=True)
        self.lib.orc_round_output(arr.ctypes.data, arr.size, _OUT_CODE[out_dtype])
        return arr

    def decode(self, bits, dtype: str) -> np.ndarray:
        """The oracle's own decode of storage elements to float64 (e2m1: each
        byte gives two elements, low nibble first; the result has twice the
        last dimension)."""
        x = _check_storage(bits, dtype, "bits")
        per = _PER_UNIT.get(dtype, 1)
        shape = x.shape[:-1] + (x.shape[-1] * per,) if x.ndim else (per,)
        out = np.zeros(shape, dtype=np.float64)
        self.lib.orc_decode_array(x.ctypes.data, x.size * per, _DTYPE_CODE[dtype], out.ctypes.data)
        return out


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def host_threads() -> int:
    return default().host_threads()


def gemm(*args, **kw):
    return default().gemm(*args, **kw)


def gemm_entries(*args, **kw):
    return default().gemm_entries(*args, **kw)


def gemm_mx(*args, **kw):
    return default().gemm_mx(*args, **kw)


def apply_epi(*args, **kw):
    return default().apply_epi(*args, **kw)


def gemm_epi(*args, **kw):
    return default().gemm_epi(*args, **kw)


def decode_scale(codes, fmt="e8m0"):
    return default().decode_scale(codes, fmt)


def decode(bits, dtype):
    return default().decode(bits, dtype)


def round_output(y, out_dtype):
    return default().round_output(y, out_dtype)
