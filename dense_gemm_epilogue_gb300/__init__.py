"""Python binding of the tg_gemm C ABI (``include/tg_gemm.h``).

Argument marshalling only: every step of the GEMM runs in the CUDA library
``_lib/libtg_gemm.so`` built from ``csrc/`` by ``build.py``.  There is no
fallback: if the library is missing, ``load()`` raises.

Pointers may be given as integers, as objects with ``data_ptr()`` (torch
tensors) or as None (NULL).  Streams may be integers (a ``cudaStream_t``),
objects with a ``cuda_stream`` attribute (``torch.cuda.Stream``) or None (the
legacy default stream).
"""

from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB as LIBRARY_PATH
from .build import build, source_hash  # noqa: F401

TG_OK = 0
TG_ERR_INVALID_VALUE = 1
TG_ERR_UNSUPPORTED = 2
TG_ERR_CUDA = 3
TG_ERR_DEVICE_TIMEOUT = 4

TG_BF16 = 0
TG_FP16 = 1
TG_TF32 = 2
TG_E4M3 = 3
TG_E5M2 = 4
TG_E2M1 = 5
TG_NVF4 = 6
DTYPE_CODES = {"bf16": TG_BF16, "fp16": TG_FP16, "tf32": TG_TF32, "e4m3": TG_E4M3,
               "e5m2": TG_E5M2, "e2m1": TG_E2M1, "nvf4": TG_NVF4}

TG_EPILOGUE_NONE = 0
TG_EPILOGUE_RELU = 1

TG_OUT_F32 = 0
TG_OUT_BF16 = 1
TG_OUT_F16 = 2
OUT_CODES = {"f32": TG_OUT_F32, "bf16": TG_OUT_BF16, "fp16": TG_OUT_F16}

# Every symbol include/tg_gemm.h declares.
EXPORTED = (
    "tg_gemm",
    "tg_gemm_ex",
    "tg_plan",
    "tg_plan_describe",
    "tg_status_string",
    "tg_check_device_status",
    "tg_set_wait_limit_ns",
    "tg_selftest_wait_timeout",
    "tg_version",
    "tg_gemm_noalloc",
    "tg_gemm_batched",
    "tg_gemm_epilogue",
    "tg_gemm_mx",
    "tg_gemm_mx_batched",
    "tg_plan_mx",
    "tg_mx_scale_bytes",
    "tg_mx_pack_scales",
    "tg_bs_scale_bytes",
    "tg_bs_pack_scales",
)


class TgError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {tg_status_string(status)} ({status})" if what else
                         f"{tg_status_string(status)} ({status})")


class tg_options(ctypes.Structure):
    _fields_ = [
        ("block_n", ctypes.c_int32),
        ("producer", ctypes.c_int32),
        ("swap_ab", ctypes.c_int32),
        ("raster_group", ctypes.c_int32),
        ("max_ctas", ctypes.c_int32),
        ("cta_pair", ctypes.c_int32),
        ("split_k", ctypes.c_int32),
        ("l2_hint", ctypes.c_int32),
        ("prefetch_k", ctypes.c_int32),
        ("multicast", ctypes.c_int32),
        ("schedule", ctypes.c_int32),
        ("reserved", ctypes.c_int32 * 1),
    ]


EPI_KINDS = {"scale": 0, "add": 1, "relu": 2, "leaky_relu": 3, "clamp": 4, "sigmoid": 5,
             "silu": 6, "gelu_tanh": 7, "bias_row": 8, "bias_col": 9}


class tg_epi_op(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int32),
        ("a", ctypes.c_float),
        ("b", ctypes.c_float),
        ("bias", ctypes.c_void_p),
    ]


class tg_plan_info(ctypes.Structure):
    _fields_ = [
        ("block_m", ctypes.c_int32),
        ("block_n", ctypes.c_int32),
        ("block_k", ctypes.c_int32),
        ("stages", ctypes.c_int32),
        ("producer", ctypes.c_int32),
        ("swap_ab", ctypes.c_int32),
        ("raster_group", ctypes.c_int32),
        ("grid", ctypes.c_int32),
        ("tiles", ctypes.c_int64),
        ("threads", ctypes.c_int32),
        ("smem_bytes", ctypes.c_int32),
        ("tmem_cols", ctypes.c_int32),
        ("vector_store", ctypes.c_int32),
        ("cta_pair", ctypes.c_int32),
        ("split_tiles", ctypes.c_int32),
        ("split_segs", ctypes.c_int32),
        ("multicast", ctypes.c_int32),
        ("stream_k", ctypes.c_int32),
        ("schedule", ctypes.c_int32),
        ("k_rotate", ctypes.c_int32),
        ("k_snake", ctypes.c_int32),
    ]


_lock = threading.Lock()
_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the built library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIBRARY_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"tg_gemm library not built ({p} missing); run "
                               "dense_gemm_epilogue_gb300.build.build() first")
        lib = ctypes.CDLL(p)
        i64, i32, f32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p
        lib.tg_gemm.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64, vp, i64, ctypes.c_int,
                                ctypes.c_int, vp]
        lib.tg_gemm.restype = ctypes.c_int
        lib.tg_gemm_ex.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64, vp, i64, ctypes.c_int,
                                   ctypes.c_int, ctypes.POINTER(tg_options), vp]
        lib.tg_gemm_ex.restype = ctypes.c_int
        lib.tg_plan.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, ctypes.c_int,
                                ctypes.POINTER(tg_options), i32, ctypes.POINTER(tg_plan_info)]
        lib.tg_plan.restype = ctypes.c_int
        lib.tg_plan_describe.argtypes = [i64, i64, i64, ctypes.c_int, i64, i64, i64, i32,
                                         ctypes.c_char_p, ctypes.c_size_t]
        lib.tg_plan_describe.restype = ctypes.c_int
        lib.tg_status_string.argtypes = [ctypes.c_int]
        lib.tg_status_string.restype = ctypes.c_char_p
        lib.tg_check_device_status.argtypes = [vp, ctypes.POINTER(i32)]
        lib.tg_check_device_status.restype = ctypes.c_int
        lib.tg_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        lib.tg_set_wait_limit_ns.restype = ctypes.c_int
        lib.tg_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
        lib.tg_selftest_wait_timeout.restype = ctypes.c_int
        lib.tg_gemm_noalloc.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64, vp, i64,
                                        ctypes.c_int, ctypes.c_int, vp]
        lib.tg_gemm_noalloc.restype = ctypes.c_int
        lib.tg_gemm_batched.argtypes = [i64, i64, i64, f32, vp, i64, i64, vp, i64, i64, vp, i64,
                                        i64, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.POINTER(tg_options), vp]
        lib.tg_gemm_batched.restype = ctypes.c_int
        lib.tg_gemm_epilogue.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64, vp, i64,
                                         ctypes.c_int, ctypes.c_int, ctypes.POINTER(tg_epi_op),
                                         i32, ctypes.POINTER(tg_options), vp]
        lib.tg_gemm_epilogue.restype = ctypes.c_int
        lib.tg_gemm_mx.argtypes = [i64, i64, i64, f32, vp, i64, vp, vp, i64, vp, vp, i64,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.POINTER(tg_options), vp]
        lib.tg_gemm_mx.restype = ctypes.c_int
        lib.tg_gemm_mx_batched.argtypes = [i64, i64, i64, f32, vp, i64, i64, vp, i64, vp, i64,
                                           i64, vp, i64, vp, i64, i64, i64, ctypes.c_int,
                                           ctypes.c_int, ctypes.POINTER(tg_epi_op), i32,
                                           ctypes.POINTER(tg_options), vp]
        lib.tg_gemm_mx_batched.restype = ctypes.c_int
        lib.tg_plan_mx.argtypes = [i64, i64, i64, i64, i64, i64, ctypes.c_int,
                                   ctypes.POINTER(tg_options), i32, ctypes.POINTER(tg_plan_info)]
        lib.tg_plan_mx.restype = ctypes.c_int
        lib.tg_mx_scale_bytes.argtypes = [i64, i64]
        lib.tg_mx_scale_bytes.restype = i64
        lib.tg_mx_pack_scales.argtypes = [i64, i64, vp, i64, vp, vp]
        lib.tg_mx_pack_scales.restype = ctypes.c_int
        lib.tg_bs_scale_bytes.argtypes = [i64, i64, ctypes.c_int]
        lib.tg_bs_scale_bytes.restype = i64
        lib.tg_bs_pack_scales.argtypes = [i64, i64, ctypes.c_int, vp, i64, vp, vp]
        lib.tg_bs_pack_scales.restype = ctypes.c_int
        lib.tg_version.argtypes = []
        lib.tg_version.restype = i32
        if path is None:
            _lib = lib
        return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError(f"cannot pass {type(x).__name__} as a pointer")


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    raise TypeError(f"cannot pass {type(s).__name__} as a stream")


def _dtype(d):
    return DTYPE_CODES[d] if isinstance(d, str) else int(d)


def _epi(e):
    if isinstance(e, str):
        return {"none": TG_EPILOGUE_NONE, "relu": TG_EPILOGUE_RELU}[e]
    if isinstance(e, bool):
        return TG_EPILOGUE_RELU if e else TG_EPILOGUE_NONE
    return int(e)


def _options(opts):
    if opts is None:
        return None
    if isinstance(opts, tg_options):
        return ctypes.byref(opts)
    o = tg_options()
    for k, v in dict(opts).items():
        if k == "reserved":
            for i, r in enumerate(v):
                o.reserved[i] = int(r)
        else:
            setattr(o, k, int(v))
    return ctypes.byref(o)


def tg_gemm(M, N, K, alpha, A, lda, B, ldb, D, ldc, in_dtype, epilogue, stream=None) -> int:
    """D = epi(alpha * A * B); returns the tg_status code (enqueue only)."""
    return load().tg_gemm(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, _ptr(D), ldc,
                          _dtype(in_dtype), _epi(epilogue), _stream(stream))


def tg_gemm_ex(M, N, K, alpha, A, lda, B, ldb, D, ldc, in_dtype, epilogue, opts=None,
               stream=None) -> int:
    """tg_gemm with planner overrides (dict of tg_options fields)."""
    return load().tg_gemm_ex(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, _ptr(D), ldc,
                             _dtype(in_dtype), _epi(epilogue), _options(opts), _stream(stream))


def tg_gemm_noalloc(M, N, K, alpha, A, lda, B, ldb, D, ldc, in_dtype, epilogue,
                    stream=None) -> int:
    """tg_gemm for callers that cannot allocate device memory (the library
    allocates nothing in this call; see include/tg_gemm.h)."""
    return load().tg_gemm_noalloc(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, _ptr(D), ldc,
                                  _dtype(in_dtype), _epi(epilogue), _stream(stream))


def tg_gemm_batched(M, N, K, alpha, A, lda, stride_a, B, ldb, stride_b, D, ldc, stride_d, batch,
                    in_dtype, out_dtype, epilogue, opts=None, stream=None) -> int:
    """Strided batch of GEMMs with an output type (f32, bf16 or fp16)."""
    out = OUT_CODES[out_dtype] if isinstance(out_dtype, str) else int(out_dtype)
    return load().tg_gemm_batched(M, N, K, alpha, _ptr(A), lda, stride_a, _ptr(B), ldb, stride_b,
                                  _ptr(D), ldc, stride_d, batch, _dtype(in_dtype), out,
                                  _epi(epilogue), _options(opts), _stream(stream))


def tg_plan(M, N, K, A, lda, B, ldb, D, ldc, in_dtype, opts=None, num_sms=0):
    """The planner's choice as a dict; raises TgError on invalid arguments."""
    info = tg_plan_info()
    st = load().tg_plan(M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(D), ldc, _dtype(in_dtype),
                        _options(opts), num_sms, ctypes.byref(info))
    if st != TG_OK:
        raise TgError(st, "tg_plan")
    return {name: getattr(info, name) for name, _ in tg_plan_info._fields_}


def tg_plan_describe(M, N, K, in_dtype, lda, ldb, ldc, num_sms=0, size=256):
    """The planner's choice as one line of text; raises TgError on invalid
    arguments or when the text does not fit in `size` bytes."""
    buf = ctypes.create_string_buffer(size)
    st = load().tg_plan_describe(M, N, K, _dtype(in_dtype), lda, ldb, ldc, num_sms, buf, size)
    if st != TG_OK:
        raise TgError(st, "tg_plan_describe")
    return buf.value.decode()


def _epi_ops(ops):
    arr = (tg_epi_op * max(len(ops), 1))()
    for q, (kind, a, b, bias) in enumerate(ops):
        arr[q].kind = EPI_KINDS[kind] if isinstance(kind, str) else int(kind)
        arr[q].a = float(a)
        arr[q].b = float(b)
        arr[q].bias = _ptr(bias)
    return arr


def tg_gemm_epilogue(M, N, K, alpha, A, lda, B, ldb, D, ldc, in_dtype, out_dtype, ops,
                     opts=None, stream=None) -> int:
    """D = out(op_n(... op_1(alpha * A B))); ops: sequence of (kind, a, b, bias)
    with kind a name of EPI_KINDS (or its code) and bias a device tensor or None."""
    out = OUT_CODES[out_dtype] if isinstance(out_dtype, str) else int(out_dtype)
    arr = _epi_ops(ops)
    return load().tg_gemm_epilogue(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, _ptr(D), ldc,
                                   _dtype(in_dtype), out, arr, len(ops), _options(opts),
                                   _stream(stream))


def tg_gemm_mx(M, N, K, alpha, A, lda, SFA, B, ldb, SFB, D, ldc, in_dtype, out_dtype, epilogue,
               opts=None, stream=None) -> int:
    """Block-scaled FP8 GEMM; SFA / SFB are scale-atom buffers (see
    include/tg_gemm.h, tg_gemm_mx)."""
    out = OUT_CODES[out_dtype] if isinstance(out_dtype, str) else int(out_dtype)
    return load().tg_gemm_mx(M, N, K, alpha, _ptr(A), lda, _ptr(SFA), _ptr(B), ldb, _ptr(SFB),
                             _ptr(D), ldc, _dtype(in_dtype), out, _epi(epilogue), _options(opts),
                             _stream(stream))


def tg_gemm_mx_batched(M, N, K, alpha, A, lda, stride_a, SFA, stride_sfa, B, ldb, stride_b, SFB,
                       stride_sfb, D, ldc, stride_d, batch, in_dtype, out_dtype, ops=(),
                       opts=None, stream=None) -> int:
    """Strided batch of block-scaled GEMMs with a composed epilogue (see
    include/tg_gemm.h, tg_gemm_mx_batched); scale strides in bytes."""
    out = OUT_CODES[out_dtype] if isinstance(out_dtype, str) else int(out_dtype)
    arr = _epi_ops(ops)
    return load().tg_gemm_mx_batched(M, N, K, alpha, _ptr(A), lda, stride_a, _ptr(SFA),
                                     stride_sfa, _ptr(B), ldb, stride_b, _ptr(SFB), stride_sfb,
                                     _ptr(D), ldc, stride_d, batch, _dtype(in_dtype), out, arr,
                                     len(ops), _options(opts), _stream(stream))


def tg_plan_mx(M, N, K, lda, ldb, ldc, in_dtype, opts=None, num_sms=0):
    """The block-scaled planner's choice as a dict; raises TgError on invalid arguments."""
    info = tg_plan_info()
    st = load().tg_plan_mx(M, N, K, lda, ldb, ldc, _dtype(in_dtype), _options(opts), num_sms,
                           ctypes.byref(info))
    if st != TG_OK:
        raise TgError(st, "tg_plan_mx")
    return {name: getattr(info, name) for name, _ in tg_plan_info._fields_}


def tg_mx_scale_bytes(rows, K) -> int:
    return int(load().tg_mx_scale_bytes(rows, K))


def tg_mx_pack_scales(rows, K, src, ld_src, dst, stream=None) -> int:
    """Row-major scale codes (device) -> scale atoms (device)."""
    return load().tg_mx_pack_scales(rows, K, _ptr(src), ld_src, _ptr(dst), _stream(stream))


def tg_bs_scale_bytes(rows, K, in_dtype) -> int:
    return int(load().tg_bs_scale_bytes(rows, K, _dtype(in_dtype)))


def tg_bs_pack_scales(rows, K, in_dtype, src, ld_src, dst, stream=None) -> int:
    """Row-major scale codes (device) -> scale atoms (device), for in_dtype's
    block size (32 K per scale; nvf4: 16)."""
    return load().tg_bs_pack_scales(rows, K, _dtype(in_dtype), _ptr(src), ld_src, _ptr(dst),
                                    _stream(stream))


def tg_status_string(status: int) -> str:
    return load().tg_status_string(int(status)).decode()


def tg_check_device_status(stream=None):
    """(status, where): synchronises the stream and reads/clears the status word."""
    where = ctypes.c_int32(0)
    st = load().tg_check_device_status(_stream(stream), ctypes.byref(where))
    return st, where.value


def tg_set_wait_limit_ns(ns: int) -> int:
    return load().tg_set_wait_limit_ns(int(ns))


def tg_selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    return load().tg_selftest_wait_timeout(int(limit_ns), _stream(stream))


def tg_version() -> int:
    return load().tg_version()


def check(status: int, what: str = "tg_gemm") -> None:
    if status != TG_OK:
        raise TgError(status, what)
