// tg_gemm_noalloc: the GEMM entry point for callers that cannot allocate
// device memory.
//
// tg_gemm allocates one word of device memory per device on its first call
// there (the status word its kernel writes when a bounded wait runs out).
// Some callers cannot let a library do that: a process whose device memory is
// all reserved up front by its own pool allocator, code that must not make
// cudaMalloc's implicit device-wide synchronisation inside a latency-critical
// loop, or code running while a stream is being captured in a mode that
// forbids cudaMalloc.  This entry point runs the same kernel with the same
// planner, but its scratch lives in a fixed file-scope __device__ array that
// the module loader places when the library is loaded, so the call itself
// allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
//
// Scratch: the array below, kNoAllocScratchBytes (256) bytes, 256-byte
// aligned, present on every device that loads the library until the process
// exits.  The kernel needs 4 bytes of it (its status word) for any M, N, K;
// a plan needing more than the array holds is rejected with
// TG_ERR_UNSUPPORTED before anything is launched.
//
// Set-up: the first call on a device (with that device current) looks up the
// array's device address with cudaGetSymbolAddress and caches it; make that
// first call before any stream capture.  Later calls on the device reuse it.
//
// Sharing: every call on a device uses the same array, which keeps what the
// last call left in it.  Each call first clears the status word on its own
// stream (cudaMemsetAsync), so calls on one stream are independent; calls
// that overlap on the GPU (different streams, concurrently) race on the word.
// The word only records a wait that ran out; this entry point does not read
// it back, and its kernels use the default 4 s wait limit.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "../../include/tg_gemm.h"
#include "tg_launch.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 256;
constexpr size_t kStatusBytes = sizeof(uint32_t);
constexpr uint64_t kNoAllocWaitLimitNs = 4000000000ull;
constexpr int kMaxDevices = 64;

// Word 0: the kernel's status word.  The rest is headroom up to the stated
// maximum.  Device code could name the array directly; host code only ever
// uses the address cudaGetSymbolAddress returns.
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocScratchBytes / sizeof(uint32_t)];

struct NoAllocDevice {
    bool ready = false;
    int sms = 0;
    uint32_t *scratch = nullptr;  // device address of g_noalloc_scratch on this device
};

std::mutex g_mutex;
NoAllocDevice g_devices[kMaxDevices];

tg_status noalloc_setup(int *dev_out, NoAllocDevice **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TG_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TG_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    NoAllocDevice &d = g_devices[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return TG_ERR_CUDA;
        if (major != 10 || minor != 3) return TG_ERR_UNSUPPORTED;
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) return TG_ERR_CUDA;
        d.scratch = static_cast<uint32_t *>(p);
        d.ready = true;
    }
    *dev_out = dev;
    *out = &d;
    return TG_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn noalloc_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Same operand description as the allocating path: dims (K, rows), byte
// stride ld * e, 128-byte rows x box_rows, 128-byte swizzle, zero fill.
bool noalloc_encode(CUtensorMap *map, tg_dtype t, const void *base, int64_t rows, int64_t k,
                    int64_t ld, int box_rows) {
    EncodeTiledFn fn = noalloc_encode_fn();
    if (!fn) return false;
    const bool fp8 = t == TG_E4M3 || t == TG_E5M2;
    const int e = t == TG_TF32 ? 4 : fp8 ? 1 : 2;
    const CUtensorMapDataType dt = t == TG_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : t == TG_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                   : fp8          ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    // Three dimensions (K, rows, one batch entry), as the kernels load.
    cuuint64_t dims[3] = {(cuuint64_t)k, (cuuint64_t)rows, 1};
    cuuint64_t strides[2] = {(cuuint64_t)(ld * e), (cuuint64_t)(ld * e)};
    cuuint32_t box[3] = {(cuuint32_t)(128 / e), (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

extern "C" tg_status tg_gemm_noalloc(int64_t M, int64_t N, int64_t K, float alpha, const void *A,
                                     int64_t lda, const void *B, int64_t ldb, float *D,
                                     int64_t ldc, tg_dtype in_dtype, tg_epilogue epilogue,
                                     void *stream_ptr) {
    if (epilogue != TG_EPILOGUE_NONE && epilogue != TG_EPILOGUE_RELU) return TG_ERR_INVALID_VALUE;
    // NULL is allowed only for an empty matrix (tg_plan reads NULL as an
    // aligned placeholder, so check it here first).
    if (M > 0 && K > 0 && A == nullptr) return TG_ERR_INVALID_VALUE;
    if (K > 0 && N > 0 && B == nullptr) return TG_ERR_INVALID_VALUE;
    if (M > 0 && N > 0 && D == nullptr) return TG_ERR_INVALID_VALUE;
    // Argument validation only (a positive SM count keeps tg_plan off CUDA).
    tg_plan_info info;
    tg_status st = tg_plan(M, N, K, A, lda, B, ldb, D, ldc, in_dtype, nullptr, 1, &info);
    if (st != TG_OK) return st;
    if (M == 0 || N == 0) return TG_OK;

    int dev = 0;
    NoAllocDevice *nd = nullptr;
    st = noalloc_setup(&dev, &nd);
    if (st != TG_OK) return st;
    if (kStatusBytes > kNoAllocScratchBytes) return TG_ERR_UNSUPPORTED;  // scratch too small
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    if (cudaMemsetAsync(nd->scratch, 0, kStatusBytes, stream) != cudaSuccess) return TG_ERR_CUDA;
    const int relu = epilogue == TG_EPILOGUE_RELU ? 1 : 0;

    if (K == 0) {
        // The empty sums, by the same fill kernel as tg_gemm (one FP32 output).
        static const tg::EpiProgram kNoOps = {};
        return tg::launch_fill_empty_sum(D, M, N, ldc, 0, 1, 0, alpha, relu, kNoOps, nd->sms,
                                         stream) == cudaSuccess
                   ? TG_OK
                   : TG_ERR_CUDA;
    }

    // No split-K tail here: it would need a workspace.
    tg_options no_split = {};
    no_split.split_k = 1;
    st = tg_plan(M, N, K, A, lda, B, ldb, D, ldc, in_dtype, &no_split, nd->sms, &info);
    if (st != TG_OK) return st;
    const bool swap = info.swap_ab != 0;
    const int64_t mk = swap ? N : M, nk = swap ? M : N;
    const void *ar = swap ? B : A;
    const void *br = swap ? A : B;
    const int64_t ldar = swap ? ldb : lda, ldbr = swap ? lda : ldb;

    tg::LaunchArgs la;
    std::memset(&la, 0, sizeof(la));
    la.block_n = info.block_n;
    la.plain_loads = info.producer == 2;
    la.pair = info.cta_pair != 0;
    la.mc = info.multicast == 2 ? 2 : 1;
    int64_t tiles = info.tiles;
    int grid = info.grid;
    if (!la.plain_loads &&
        !(noalloc_encode(&la.map_a, in_dtype, ar, mk, K, ldar,
                         la.pair && la.mc == 2 ? tg::BLOCK_M / 2 : tg::BLOCK_M) &&
          noalloc_encode(&la.map_b, in_dtype, br, nk, K, ldbr,
                         la.pair ? info.block_n / 2 : info.block_n))) {
        // Shapes the TMA unit cannot describe: single-CTA tiles, plain loads.
        la.plain_loads = true;
        la.pair = false;
        la.mc = 1;
        tiles = cdiv(mk, tg::BLOCK_M) * cdiv(nk, info.block_n);
        grid = (int)(tiles < nd->sms ? tiles : nd->sms);
    }
    tg::GemmParams &p = la.p;
    p.m = (int32_t)mk;
    p.n = (int32_t)nk;
    p.k = (int32_t)K;
    p.num_m_blocks = (int32_t)cdiv(mk, la.pair ? 2 * tg::BLOCK_M : tg::BLOCK_M);
    p.num_n_blocks = (int32_t)cdiv(cdiv(nk, info.block_n), la.mc);
    p.num_k_blocks = (int32_t)cdiv(K, info.block_k);
    p.raster_group = info.raster_group;
    p.relu = relu;
    p.num_tiles = tiles;
    p.tiles_per_batch = tiles;
    p.batch = 1;
    p.out_fmt = 0;
    p.alpha = alpha;
    p.vector_store = info.vector_store;
    p.d = D;
    p.d_row_stride = swap ? ldc : 1;
    p.d_col_stride = swap ? 1 : ldc;
    p.a_ptr = ar;
    p.b_ptr = br;
    p.lda = ldar;
    p.ldb = ldbr;
    p.status = nd->scratch;
    p.wait_limit_ns = kNoAllocWaitLimitNs;
    p.split_max = 1;  // no split-K tail: it would need a workspace
    la.grid = grid;
    la.device = dev;
    la.stream = stream;

    cudaError_t e;
    if (in_dtype == TG_BF16) e = tg::launch_bf16(la);
    else if (in_dtype == TG_FP16) e = tg::launch_fp16(la);
    else if (in_dtype == TG_E4M3) e = tg::launch_e4m3(la);
    else if (in_dtype == TG_E5M2) e = tg::launch_e5m2(la);
    else e = tg::launch_tf32(la);
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}
