"""Child process of tests/test_zz_no_alloc.py: does tg_gemm_noalloc allocate
device memory?

Run as ``python tests/noalloc_probe.py``; prints one JSON line.  It uses no
torch: device buffers come from the CUDA runtime through ctypes, each
rounded up to whole 2 MiB pages, so that the only device allocations in the
process are the ones this script makes on purpose and whatever the library
makes.  The device's free memory (cudaMemGetInfo) is read around the calls:

1. a warm-up pass of tg_gemm_noalloc over every case on the legacy default
   stream (the set-up call, the kernels' first launches);
2. ``free_before``; two passes of tg_gemm_noalloc over every case on a
   stream created before step 1; ``free_after``;
3. the positive control: the allocating entry point, tg_gemm, on the same
   stream with a shape it splits along K, which allocates its per-stream
   workspace (about 20 MB); ``free_control``.

The parent test requires free_after == free_before and free_control well
below free_after (the measurement does see an allocation of that kind).
"""

from __future__ import annotations

import ctypes
import glob
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import seeded_inputs as si  # noqa: E402

PAGE = 2 << 20

# Every planner branch the entry point can take, and the K = 0 fill.
CASES = [
    si.Workload("tma_single", 1000, 777, 300, "bf16", 1.5, True, 71, "uniform", ldc=1004),
    si.WORKLOADS["c1_bf16_65x97x73"],                      # plain loads
    si.Workload("swap", 40, 900, 200, "fp16", -0.5, False, 72, "normal", scale=0.1, ldc=44),
    si.Workload("unsplit", 600, 900, 2048, "bf16", 1.0, True, 74, "normal", ldc=600),
    si.Workload("pair", 1999, 1501, 1000, "bf16", 0.75, True, 76, "normal", ldc=2004),
    si.Workload("multicast", 4000, 4900, 1000, "bf16", 1.0, True, 75, "uniform", lda=1008,
                ldb=1008, ldc=4004),
    si.Workload("tf32", 300, 200, 96, "tf32", 1.0, False, 73, "uniform", lo=0.0),
    si.Workload("k0", 70, 90, 0, "bf16", -2.0, True, 1, "uniform", lda=1, ldb=1, ldc=72),
]
# A shape the allocating entry point splits along K (its workspace).
SPLIT = si.Workload("split", 600, 900, 2048, "bf16", 1.0, True, 74, "normal", ldc=600)


def cudart() -> ctypes.CDLL:
    """The shared CUDA runtime of the toolkit (or of the CUDA wheels)."""
    cands = []
    for base in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if base:
            cands += sorted(glob.glob(os.path.join(base, "lib64", "libcudart.so*")))
            cands += sorted(glob.glob(os.path.join(base, "targets", "*", "lib", "libcudart.so*")))
    for p in sys.path:
        cands += sorted(glob.glob(os.path.join(p, "nvidia", "cuda_runtime", "lib",
                                               "libcudart.so*")))
    for c in cands:
        try:
            return ctypes.CDLL(c)
        except OSError:
            continue
    raise RuntimeError("no libcudart.so found")


class Runtime:
    def __init__(self):
        self.rt = cudart()
        self.rt.cudaMalloc.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t]
        self.rt.cudaMemcpy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                       ctypes.c_int]
        self.rt.cudaMemGetInfo.argtypes = [ctypes.POINTER(ctypes.c_size_t)] * 2
        self.rt.cudaStreamCreate.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
        self.rt.cudaStreamSynchronize.argtypes = [ctypes.c_void_p]

    def ok(self, rc, what):
        if rc != 0:
            raise RuntimeError(f"{what} failed with CUDA error {rc}")

    def malloc_pages(self, nbytes: int) -> int:
        p = ctypes.c_void_p()
        self.ok(self.rt.cudaMalloc(ctypes.byref(p), max(PAGE, -(-nbytes // PAGE) * PAGE)),
                "cudaMalloc")
        return p.value

    def upload(self, x: np.ndarray) -> int:
        x = np.ascontiguousarray(x)
        d = self.malloc_pages(x.nbytes)
        self.ok(self.rt.cudaMemcpy(d, x.ctypes.data, x.nbytes, 1), "cudaMemcpy")
        return d

    def free_bytes(self) -> int:
        self.ok(self.rt.cudaDeviceSynchronize(), "cudaDeviceSynchronize")
        f, t = ctypes.c_size_t(), ctypes.c_size_t()
        self.ok(self.rt.cudaMemGetInfo(ctypes.byref(f), ctypes.byref(t)), "cudaMemGetInfo")
        return f.value


def main() -> int:
    import dense_gemm_epilogue_gb300 as tg

    cu = Runtime()
    cu.ok(cu.rt.cudaSetDevice(0), "cudaSetDevice")
    cu.ok(cu.rt.cudaFree(None), "context creation")
    stream = ctypes.c_void_p()
    cu.ok(cu.rt.cudaStreamCreate(ctypes.byref(stream)), "cudaStreamCreate")
    lib = tg.load()

    bufs = []
    for w in CASES + [SPLIT]:
        A, B = si.make_operands(w)
        bufs.append((w, cu.upload(A), cu.upload(B), cu.upload(si.make_output(w))))

    def noalloc_pass(st):
        for w, dA, dB, dD in bufs[:-1]:
            lda, ldb, ldc = w.strides
            rc = lib.tg_gemm_noalloc(w.M, w.N, w.K, w.alpha, dA, lda, dB, ldb, dD, ldc,
                                     tg.DTYPE_CODES[w.dtype], int(w.relu), st)
            if rc != tg.TG_OK:
                raise RuntimeError(f"tg_gemm_noalloc({w.name}) returned {rc}")

    noalloc_pass(None)
    free_before = cu.free_bytes()
    for _ in range(2):
        noalloc_pass(stream)
    cu.ok(cu.rt.cudaStreamSynchronize(stream), "cudaStreamSynchronize")
    free_after = cu.free_bytes()

    w, dA, dB, dD = bufs[-1]
    lda, ldb, ldc = w.strides
    plan = tg.tg_plan(w.M, w.N, w.K, dA, lda, dB, ldb, dD, ldc, w.dtype, None, 152)
    rc = lib.tg_gemm(w.M, w.N, w.K, w.alpha, dA, lda, dB, ldb, dD, ldc, tg.DTYPE_CODES[w.dtype],
                     int(w.relu), stream)
    if rc != tg.TG_OK:
        raise RuntimeError(f"tg_gemm({w.name}) returned {rc}")
    free_control = cu.free_bytes()
    print(json.dumps({"free_before": free_before, "free_after": free_after,
                      "free_control": free_control, "control_split_segs": plan["split_segs"],
                      "cases": [w.name for w in CASES]}), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
