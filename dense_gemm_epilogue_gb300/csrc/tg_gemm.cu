// C-ABI front end of tg_gemm: argument validation, the host planner, TMA
// tensor-map encoding, per-device state and kernel launch.
//
// The planner follows "Walk through GEMM" section 1 "Choose the work and the
// storage separately": the host picks a compiled tile configuration from the
// problem's shape, while dimensions and leading strides stay runtime kernel
// arguments.  Host validation mirrors section 3 "Copy one K stage" (the host
// checks layouts; the caller is responsible for allocation bounds).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/tg_gemm.h"
#include "tg_launch.h"

namespace tg {

// D = epi(alpha * 0) over every M x N output of the batch: the K == 0 case
// (empty sums), in the output format.  Each block covers 1024 rows (M is
// contiguous in D; four rows per thread) of one column, then steps over the
// batch's columns by the grid's y size; the column and batch indices advance
// without a division per element.
__global__ void tg_fill_empty_sum_kernel(void *d, int64_t m, int64_t n, int64_t ldc,
                                         int64_t stride_d, int64_t batch, int out_fmt, float alpha,
                                         int relu, const EpiProgram prog) {
    const float v0 = apply_epilogue(0.0f, alpha, relu);
    const int64_t i0 = blockIdx.x * 1024 + threadIdx.x;
    int64_t b = blockIdx.y / n, j = blockIdx.y - (blockIdx.y / n) * n;
    const int64_t bstep = gridDim.y / n, jstep = gridDim.y - bstep * n;
    for (; b < batch;) {
        const int64_t base = b * stride_d + j * ldc;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int64_t i = i0 + 256 * r;
            if (i < m) {
                float v = v0;
                for (int q = 0; q < prog.n; ++q) v = epi_op(prog.op[q], v, i, j);
                if (out_fmt == 0) static_cast<float *>(d)[base + i] = v;
                else if (out_fmt == 1) static_cast<unsigned short *>(d)[base + i] = OutFormat<1>::cvt(v);
                else static_cast<unsigned short *>(d)[base + i] = OutFormat<2>::cvt(v);
            }
        }
        b += bstep;
        j += jstep;
        if (j >= n) {
            j -= n;
            ++b;
        }
    }
}

// Grid of the K == 0 fill: 1024 rows per block in x; in y, enough column
// steps for about 16 blocks per SM (each block then loops over columns).
static dim3 fill_grid(int64_t m, int64_t cols, int sms) {
    const int64_t gx = (m + 1023) / 1024;
    int64_t gy = ((int64_t)sms * 16 + gx - 1) / gx;
    if (gy > cols) gy = cols;
    if (gy > 65535) gy = 65535;
    return dim3((unsigned)gx, (unsigned)(gy > 0 ? gy : 1), 1);
}

cudaError_t launch_fill_empty_sum(void *d, int64_t m, int64_t n, int64_t ldc, int64_t stride_d,
                                  int64_t batch, int out_fmt, float alpha, int relu,
                                  const EpiProgram &prog, int sms, cudaStream_t stream) {
    tg_fill_empty_sum_kernel<<<fill_grid(m, n * batch, sms), 256, 0, stream>>>(
        d, m, n, ldc, stride_d, batch, out_fmt, alpha, relu, prog);
    return cudaGetLastError();
}

// One thread waits on a barrier that nothing completes; the bounded wait must
// run out, record SITE_SELFTEST and return.
__global__ void tg_selftest_wait_kernel(uint32_t *status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t barrier_word;
    __shared__ int abort_word;
    if (threadIdx.x == 0) {
        const uint32_t b = smem_u32(&barrier_word);
        mbar_init(b, 1);
        abort_word = 0;
        fence_mbar_init();
        const WaitCtl ctl{reinterpret_cast<volatile int *>(&abort_word), status, limit_ns};
        wait_phase(b, 0, ctl, SITE_SELFTEST);
    }
}

// Scale atoms from row-major scales: dst byte o of atom (rb, kg) holds the
// scale of row rb*128 + ((o % 512) % 16) / 4 * 32 + (o % 512) / 16 and block
// kg*4 + o % 4 (zero outside the rows x blocks given).
__global__ void tg_mx_pack_scales_kernel(const uint8_t *src, int64_t rows, int64_t kblocks,
                                         int64_t ld_src, int64_t kgroups, int64_t total,
                                         uint8_t *dst) {
    for (int64_t o = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; o < total;
         o += (int64_t)gridDim.x * blockDim.x) {
        const int64_t atom = o >> 9, w = o & 511;
        const int64_t rb = atom / kgroups, kg = atom - rb * kgroups;
        const int64_t r = rb * 128 + ((w & 15) >> 2) * 32 + (w >> 4);
        const int64_t kb = kg * 4 + (w & 3);
        dst[o] = (r < rows && kb < kblocks) ? src[r * ld_src + kb] : (uint8_t)0;
    }
}

}  // namespace tg

namespace {

using tg::Config;
using tg::Kind;

constexpr int32_t kVersion = 100;  // 0.1.0
constexpr uint64_t kDefaultWaitLimitNs = 4000000000ull;
constexpr int kMaxDevices = 64;

std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitLimitNs};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int elem_bytes(tg_dtype t) {
    return t == TG_TF32 ? 4 : (t == TG_E4M3 || t == TG_E5M2) ? 1 : 2;
}

// Packed 4-bit floats (two per byte), with either scaling.
bool is_fp4(tg_dtype t) { return t == TG_E2M1 || t == TG_NVF4; }

// K elements per pipeline stage: one 128-byte swizzle row of the type
// (packed FP4: 256).
int block_k(tg_dtype t) { return is_fp4(t) ? 256 : 128 / elem_bytes(t); }

// K elements per block scale (block-scaled types).
int scale_k(tg_dtype t) { return t == TG_NVF4 ? 16 : 32; }

bool known_dtype(tg_dtype t) {
    return t == TG_BF16 || t == TG_FP16 || t == TG_TF32 || t == TG_E4M3 || t == TG_E5M2;
}

struct DeviceState {
    bool ready = false;
    int sms = 0;
    int cc_major = 0, cc_minor = 0;
    uint32_t *status = nullptr;  // one word of device memory owned by the library
};

std::mutex g_dev_mutex;
DeviceState g_dev[kMaxDevices];

// Split-K workspace of one (device, stream): room for `tiles` partial
// 256 x 256 FP32 pair tiles; ready flags (four per tile: one per segment and
// tile half of a two-segment exchange) and the ticket counter after them, all
// kept at zero between launches by the kernel itself.
constexpr int64_t kFlagsPerTile = 4;
constexpr int64_t kFlagWordsExtra = 32;
int64_t flag_words(int64_t tiles) { return kFlagsPerTile * tiles + kFlagWordsExtra; }
uint32_t *ticket_counter(uint32_t *flags, int64_t tiles) { return flags + kFlagsPerTile * tiles; }

struct Workspace {
    int device;
    cudaStream_t stream;
    float *ws;
    uint32_t *flags;
    int64_t tiles;
};
std::mutex g_ws_mutex;
std::vector<Workspace> g_ws;

constexpr int64_t kPairTileFloats = 256 * 256;

tg_status workspace_for(int dev, cudaStream_t stream, int64_t tiles, Workspace *out) {
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    for (Workspace &w : g_ws) {
        if (w.device == dev && w.stream == stream && w.tiles >= tiles) {
            *out = w;
            return TG_OK;
        }
    }
    Workspace w{dev, stream, nullptr, nullptr, tiles};
    if (cudaMalloc(&w.ws, sizeof(float) * kPairTileFloats * tiles) != cudaSuccess) return TG_ERR_CUDA;
    if (cudaMalloc(&w.flags, sizeof(uint32_t) * flag_words(tiles)) != cudaSuccess) {
        cudaFree(w.ws);
        return TG_ERR_CUDA;
    }
    if (cudaMemset(w.flags, 0, sizeof(uint32_t) * flag_words(tiles)) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaFree(w.flags);
        cudaFree(w.ws);
        return TG_ERR_CUDA;
    }
    // A smaller workspace of the same stream stays allocated (it may still be
    // in use by queued work); the larger one replaces it for later calls.
    for (Workspace &old : g_ws)
        if (old.device == dev && old.stream == stream) old.stream = reinterpret_cast<cudaStream_t>(~uintptr_t(0));
    g_ws.push_back(w);
    *out = w;
    return TG_OK;
}

// After a bounded wait ran out, flags may be left raised and a ticket counter
// away from zero: clear them all.
tg_status reset_workspace_flags(int dev) {
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    for (Workspace &w : g_ws)
        if (w.device == dev && cudaMemset(w.flags, 0, sizeof(uint32_t) * flag_words(w.tiles)) != cudaSuccess)
            return TG_ERR_CUDA;
    return TG_OK;
}

// Per-device set-up on first use: device attributes and the status word.
tg_status device_state(int *dev_out, DeviceState **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TG_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TG_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceState &s = g_dev[dev];
    if (!s.ready) {
        if (cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&s.cc_major, cudaDevAttrComputeCapabilityMajor, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&s.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) !=
                cudaSuccess)
            return TG_ERR_CUDA;
        if (s.cc_major != 10 || s.cc_minor != 3) return TG_ERR_UNSUPPORTED;
        if (cudaMalloc(&s.status, sizeof(uint32_t)) != cudaSuccess) return TG_ERR_CUDA;
        if (cudaMemset(s.status, 0, sizeof(uint32_t)) != cudaSuccess ||
            cudaDeviceSynchronize() != cudaSuccess) {
            cudaFree(s.status);
            s.status = nullptr;
            return TG_ERR_CUDA;
        }
        s.ready = true;
    }
    *dev_out = dev;
    *out = &s;
    return TG_OK;
}

// ------------------------------------------------------------------ planner

// Split-K tail: the kernel cuts each of the last R = tiles mod pairs tiles
// into S = min(pairs / R, split_max, K blocks / 8) K segments (see
// tg_kernel_pair.cuh); the host mirrors the rule to size and report it.
// By default: up to kDefaultSplitMax segments when there are fewer tiles
// than pairs; with a wave or more, two segments when the last wave is at most
// half full (the two exchange halves of their partial sums, which measured
// 1-3 % faster than whole tiles at 4096^3 and 8192^3 in bursts of launches;
// an earlier one-sided fix-up measured no gain under sustained load).
constexpr int kDefaultSplitMax = 8;

// The ticket schedule is the planner's choice from this many waves of
// CTA-pair tiles up (see make_plan).
constexpr int64_t kTicketMinWaves = 6;

// Stream-K (single-CTA tiles): a CTA's share spans at least this many K
// blocks, so that its MMA work outweighs writing or reading one partial tile.
constexpr int64_t kStreamKMinBlocks = 8;

// Rotated K order (single-CTA, one wave of whole tiles): the largest
// operand shared by several tiles that the rotation still keeps in L2.
constexpr int64_t kRotateSharedBytes = 32ll << 20;
// ... and the shortest K loop (in K blocks) it is used for: it matters for
// long streaming loops only.
constexpr int64_t kRotateMinBlocks = 16;

// Planner cost of finishing a K-split tile (flag wait, partial-sum round
// trip through L2), in the planner's cost units: about 4 us measured, some
// 22 K blocks of a 128 x 64 tile.  Splitting therefore pays only for long
// K loops (1024^3 runs 8.5 us unsplit, 11.6-12.6 us split either way).
constexpr int64_t kFixupLatency = 5632;

void split_rule(int64_t tiles, int64_t pairs, int64_t nkb, int split_max, int64_t ws_tiles,
                int64_t *rem_out, int *segs_out) {
    int64_t rem = tiles % pairs, segs = 1;
    if (split_max > 1 && rem > 0) {
        segs = pairs / rem;
        if (segs > split_max) segs = split_max;
        if (segs > nkb / tg::SPLIT_MIN_KBLOCKS) segs = nkb / tg::SPLIT_MIN_KBLOCKS;
        if (segs < 2 || rem * (segs - 1) > ws_tiles) segs = 1;
    }
    *rem_out = segs > 1 ? rem : 0;
    *segs_out = (int)segs;
}

// One call's problem: a batch of `batch` GEMMs of the same shape.
struct Problem {
    int64_t M, N, K;
    float alpha;
    const void *A;
    int64_t lda, sa;  // leading stride, batch stride (elements of the input type)
    const void *B;
    int64_t ldb, sb;
    void *D;
    int64_t ldc, sd;  // elements of the output type
    int64_t batch;
    tg_dtype t;
    int out_fmt;      // 0 FP32, 1 BF16, 2 FP16
    int relu;
};

int out_bytes(int out_fmt) { return out_fmt == 0 ? 4 : 2; }

struct Plan {
    bool pair = false;  // CTA-pair kernel (256-row tiles over a 2-CTA cluster)
    int mc = 1;         // pair kernel: pairs per cluster (2: A rows multicast)
    int split_max = 1;  // K segments allowed per tail tile (pair kernel only)
    bool dynamic = false;  // pair kernel: one cluster per tile, launch-control stealing
    bool stream_k = false; // single-CTA kernel: each CTA a contiguous share of all K iterations
    bool ticket = false;   // pair kernel: first unit static, later units claimed from a counter
    int64_t split_tiles = 0;
    int split_segs = 1;
    bool swap = false;
    int block_n = 0;
    int producer = 0;  // 1 TMA, 2 plain loads
    int stages = 0;
    int group = 0;
    int grid = 0;
    int64_t tiles = 0;            // all tiles of the batch
    int64_t tiles_per_batch = 0;
    int threads = 0;
    int smem = 0;
    int tmem_cols = 0;
    bool vector_store = false;
    bool k_rotate = false;   // single-CTA whole tiles: rotated K order per tile
    bool k_snake = false;    // CTA-pair tiles: odd waves walk K in descending order
    int64_t mk = 0, nk = 0;  // role-space rows and cols
};

template <Kind KD>
void config_numbers(int bn, int *stages, int *smem, int *threads, int *tmem) {
    switch (bn) {
#define TG_CASE(BN)                                   \
    case BN:                                          \
        *stages = Config<KD, BN>::STAGES;             \
        *smem = Config<KD, BN>::SMEM_BYTES;           \
        *threads = Config<KD, BN>::NUM_THREADS;       \
        *tmem = Config<KD, BN>::TMEM_COLS;            \
        break;
        TG_CASE(64)
        TG_CASE(128)
        TG_CASE(256)
#undef TG_CASE
    default:
        *stages = *smem = *threads = *tmem = 0;
    }
}

template <Kind KD>
void pair_numbers(int bn, int *stages, int *smem, int *threads, int *tmem) {
    if (bn == 256) {
        using C = tg::PairConfig<KD, 256>;
        *stages = C::STAGES; *smem = C::SMEM_BYTES; *threads = C::NUM_THREADS; *tmem = C::TMEM_COLS;
    } else {
        using C = tg::PairConfig<KD, 128>;
        *stages = C::STAGES; *smem = C::SMEM_BYTES; *threads = C::NUM_THREADS; *tmem = C::TMEM_COLS;
    }
}

void config_numbers_for(tg_dtype t, int bn, int *stages, int *smem, int *threads, int *tmem) {
    if (t == TG_BF16) config_numbers<Kind::BF16>(bn, stages, smem, threads, tmem);
    else if (t == TG_FP16) config_numbers<Kind::FP16>(bn, stages, smem, threads, tmem);
    else if (t == TG_E4M3) config_numbers<Kind::E4M3>(bn, stages, smem, threads, tmem);
    else if (t == TG_E5M2) config_numbers<Kind::E5M2>(bn, stages, smem, threads, tmem);
    else config_numbers<Kind::TF32>(bn, stages, smem, threads, tmem);
}

bool tma_legal(const void *p, int64_t ld, int esize) {
    const uint64_t stride = (uint64_t)ld * (uint64_t)esize;
    return ((uintptr_t)p % 16) == 0 && stride % 16 == 0 && stride < (1ull << 40);
}

// A batch stride the TMA can address as a third tensor dimension (a zero
// stride, one operand for every batch entry, needs no dimension at all).
bool tma_batch_legal(int64_t stride, int esize, int64_t batch) {
    if (batch <= 1 || stride == 0) return true;
    const uint64_t bytes = (uint64_t)stride * (uint64_t)esize;
    return bytes % 16 == 0 && bytes < (1ull << 40);
}

tg_status validate(const Problem &q, const tg_options *o) {
    const tg_dtype t = q.t;
    const int64_t M = q.M, N = q.N, K = q.K;
    if (!known_dtype(t)) return TG_ERR_INVALID_VALUE;
    if (q.out_fmt < 0 || q.out_fmt > 2) return TG_ERR_INVALID_VALUE;
    if (M < 0 || N < 0 || K < 0 || q.batch < 0) return TG_ERR_INVALID_VALUE;
    if (q.lda < (K > 1 ? K : 1) || q.ldb < (K > 1 ? K : 1) || q.ldc < (M > 1 ? M : 1))
        return TG_ERR_INVALID_VALUE;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX || q.batch > INT32_MAX)
        return TG_ERR_UNSUPPORTED;
    if (q.batch > 1) {
        // Operands may be shared by all batch entries (stride 0); outputs may not.
        if (q.sa < 0 || q.sb < 0) return TG_ERR_INVALID_VALUE;
        if (M * N > 0 && q.sd < q.ldc * N) return TG_ERR_INVALID_VALUE;
    }
    const int e = elem_bytes(t), eo = out_bytes(q.out_fmt);
    if (M * K > 0 && (q.A == nullptr || (uintptr_t)q.A % e)) return TG_ERR_INVALID_VALUE;
    if (K * N > 0 && (q.B == nullptr || (uintptr_t)q.B % e)) return TG_ERR_INVALID_VALUE;
    if (M * N > 0 && (q.D == nullptr || (uintptr_t)q.D % eo)) return TG_ERR_INVALID_VALUE;
    if (o) {
        if (o->block_n != 0 && o->block_n != 64 && o->block_n != 128 && o->block_n != 256)
            return TG_ERR_INVALID_VALUE;
        if (o->producer < 0 || o->producer > 2) return TG_ERR_INVALID_VALUE;
        if (o->swap_ab < 0 || o->swap_ab > 2) return TG_ERR_INVALID_VALUE;
        if (o->raster_group < 0 || o->max_ctas < 0) return TG_ERR_INVALID_VALUE;
        if (o->cta_pair < 0 || o->cta_pair > 2) return TG_ERR_INVALID_VALUE;
        if (o->split_k < 0 || o->split_k > 64) return TG_ERR_INVALID_VALUE;
        if (o->l2_hint < 0 || o->l2_hint > 2) return TG_ERR_INVALID_VALUE;
        if (o->prefetch_k < -1 || o->prefetch_k > 64) return TG_ERR_INVALID_VALUE;
        if (o->multicast < 0 || o->multicast > 2) return TG_ERR_INVALID_VALUE;
        if (o->schedule < 0 || o->schedule > 4 || o->reserved[0]) return TG_ERR_INVALID_VALUE;
        // Tickets run CTA-pair tiles, one pair per cluster, with the workspace.
        if (o->schedule == 4 && (o->cta_pair == 1 || o->multicast == 2 || o->split_k == 1))
            return TG_ERR_INVALID_VALUE;
        // Stream-K runs single-CTA tiles and splits K by definition.
        if (o->schedule == 3 && (o->cta_pair == 2 || o->multicast == 2 || o->split_k == 1))
            return TG_ERR_INVALID_VALUE;
        if (o->multicast == 2 && o->cta_pair == 1) return TG_ERR_INVALID_VALUE;
        // The dynamic schedule runs CTA-pair tiles, one pair per cluster, whole tiles.
        if (o->schedule == 2 && (o->cta_pair == 1 || o->multicast == 2 || o->split_k > 1))
            return TG_ERR_INVALID_VALUE;
        // Overrides that cannot apply to this problem.
        const bool legal = tma_legal(q.A, q.lda, e) && tma_legal(q.B, q.ldb, e) &&
                           tma_batch_legal(q.sa, e, q.batch) && tma_batch_legal(q.sb, e, q.batch);
        if (o->producer == 1 && !legal) return TG_ERR_INVALID_VALUE;
        if (o->cta_pair == 2 && (t == TG_TF32 || !legal || o->producer == 2 || o->block_n == 64))
            return TG_ERR_INVALID_VALUE;
    }
    return TG_OK;
}

// Plan a problem with M, N, K, batch > 0 (arguments already validated).
tg_status make_plan(const Problem &q, const tg_options *o, int sms, Plan *plan) {
    static const tg_options kNone = {};
    if (!o) o = &kNone;
    const int64_t M = q.M, N = q.N, K = q.K;
    const tg_dtype t = q.t;
    Plan p;
    // Fill the 128-row MMA dimension: a short M with a long N runs with the
    // operand roles swapped (both are K-major, so nothing is transposed).
    if (o->swap_ab == 1) p.swap = false;
    else if (o->swap_ab == 2) p.swap = true;
    else p.swap = (M < tg::BLOCK_M) && (N >= tg::BLOCK_M) && (N >= 2 * M);
    p.mk = p.swap ? N : M;
    p.nk = p.swap ? M : N;

    const int e = elem_bytes(t);
    const bool legal = tma_legal(q.A, q.lda, e) && tma_legal(q.B, q.ldb, e) &&
                       tma_batch_legal(q.sa, e, q.batch) && tma_batch_legal(q.sb, e, q.batch);
    if (o->producer == 1 && !legal) return TG_ERR_INVALID_VALUE;
    p.producer = o->producer ? o->producer : (legal ? 1 : 2);

    // Tile shape and schedule: the candidate with the smallest estimated time,
    // (K blocks run in sequence by one CTA or pair) x (cycles per K block) +
    // the fix-up of K-split tiles.  Per 16-wide K step an SM's tensor core
    // needs BN/2 cycles (128 rows each), and its shared memory moves the A and
    // B bytes twice (TMA write, tensor-core read) at about 128 B/cycle: 64 +
    // BN/2 cycles for a single-CTA tile, 64 + BN/4 when a CTA pair splits B;
    // a K step costs the larger of the two, and a K block is four steps
    // (8-bit kinds take 32 elements per 32-byte step at twice the rate, TF32 8
    // per 32 bytes at half, so the same per-byte costs apply).  A K-split tile
    // (pair split tail, stream-K) adds kFixupLatency and 8 x BN cycles per
    // partial tile its finisher reads (128 x BN FP32 at about 64 B/cycle).
    // Calibrated on 1024^2 x 8192, 2048 x 512 x 16384, 512 x 2048 x 4096,
    // 256^2 x 65536, 1024^3, 4096 x 128 x 8192, 128 x 4096 x 2048 and
    // 256 x 128 x 512 (TF32): on each it picks the measured fastest
    // candidate or one within 3 % of it.  Pair tiles need 16-bit or 8-bit
    // operands on TMA.
    const bool pair_ok = t != TG_TF32 && p.producer == 1;
    // The dynamic schedule runs CTA-pair tiles only; stream-K single-CTA tiles.
    const bool force_pair = o->cta_pair == 2 || o->schedule == 2 || o->schedule == 4;
    const bool force_single = o->cta_pair == 1 || o->schedule == 3;
    if (force_pair && !pair_ok) return TG_ERR_INVALID_VALUE;
    if (force_pair && o->block_n == 64) return TG_ERR_INVALID_VALUE;
    // Pair tiles need a few K blocks to fill their 7-stage ring.
    const int64_t nkb = ceil_div(K, block_k(t));
    const bool pair_auto = pair_ok && nkb >= 8;
    struct Cand { bool pair; int bn; };
    Cand cands[5];
    int nc = 0;
    // Ties go to single-CTA tiles, then to the wider tile.
    for (int bn : {256, 128, 64})
        if ((!o->block_n || o->block_n == bn) && !force_pair) cands[nc++] = {false, bn};
    for (int bn : {256, 128})
        if ((!o->block_n || o->block_n == bn) && !force_single &&
            (force_pair ? pair_ok : pair_auto))
            cands[nc++] = {true, bn};
    int64_t cap = sms;
    if (o->max_ctas && cap > o->max_ctas) cap = o->max_ctas;
    if (cap < 1) cap = 1;
    const bool sk_ok = o->split_k != 1 && (o->schedule == 0 || o->schedule == 3);
    int64_t best = -1;
    for (int i = 0; i < nc; ++i) {
        const Cand c = cands[i];
        const int rows = c.pair ? 2 * tg::BLOCK_M : tg::BLOCK_M;
        const int64_t tiles = q.batch * ceil_div(p.mk, rows) * ceil_div(p.nk, c.bn);
        int64_t slots = c.pair ? cap / 2 : cap;
        if (slots < 1) slots = 1;
        const int64_t mma = c.bn / 2;
        // TF32 stages pass through shared memory twice more (narrowed in place
        // by other warps, one more barrier hop per stage): three times the cost.
        const int64_t smem = (c.pair ? 64 + c.bn / 4 : 64 + c.bn / 2) * (t == TG_TF32 ? 3 : 1);
        const int64_t kb_cost = 4 * (mma > smem ? mma : smem);
        int64_t chain = ceil_div(tiles, slots) * nkb, fix = 0;
        if (c.pair && tiles < slots && o->split_k != 1 && o->schedule != 2) {
            int64_t segs = slots / tiles;
            const int64_t smax = o->split_k ? o->split_k : kDefaultSplitMax;
            if (segs > smax) segs = smax;
            if (segs > nkb / tg::SPLIT_MIN_KBLOCKS) segs = nkb / tg::SPLIT_MIN_KBLOCKS;
            if (segs > 1) {
                chain = ceil_div(nkb, segs);
                fix = kFixupLatency + (segs - 1) * 8 * c.bn;
            }
        }
        int64_t est = chain * kb_cost + fix;
        bool sk = false;
        if (!c.pair && sk_ok) {
            const int64_t iters = tiles * nkb;
            int64_t g = iters / kStreamKMinBlocks;
            if (g > cap) g = cap;
            if (o->schedule == 3 || (tiles < cap && g > tiles)) {
                if (g < 1) g = 1;
                // CTAs over one tile: nkb / share when the shares line up
                // with the tiles, one more when they do not.
                int64_t share = iters / g;  // K blocks per CTA (at least)
                if (share < 1) share = 1;
                const int64_t segs =
                    ceil_div(nkb, share) + ((iters % g) || (nkb % share) ? 1 : 0);
                const int64_t est_sk = ceil_div(iters, g) * kb_cost + kFixupLatency +
                                       (segs - 1) * 8 * c.bn;
                if (o->schedule == 3 || est_sk < est) {
                    est = est_sk;
                    sk = true;
                }
            }
        }
        if (best < 0 || est < best) {
            best = est;
            p.pair = c.pair;
            p.block_n = c.bn;
            p.stream_k = sk;
        }
    }
    const int rows = p.pair ? 2 * tg::BLOCK_M : tg::BLOCK_M;
    const int64_t mblocks = ceil_div(p.mk, rows);
    const int64_t nblocks = ceil_div(p.nk, p.block_n);
    // Two pairs per cluster share their A rows by multicast (a quarter less
    // L2-to-SM traffic per CTA); a cluster then covers two N blocks.  The
    // planner turns it on for short K loops (at most 32 K blocks) over several
    // waves of tiles, where each tile's loads, not its MMAs, set the pace:
    // 8191x4097x1000 ran 8 % faster, 4096^3 the same, 8192^3 4 % slower.
    const bool mc_auto = o->multicast == 0 && o->schedule != 2 && o->schedule != 4 &&
                         ceil_div(K, block_k(t)) <= 32 && mblocks * nblocks >= 4 * (sms / 2);
    if (p.pair) p.mc = ((o->multicast == 2 || mc_auto) && nblocks >= 2) ? 2 : 1;
    if (o->multicast == 2 && p.pair && p.mc != 2) return TG_ERR_INVALID_VALUE;
    p.tiles_per_batch = mblocks * ceil_div(nblocks, p.mc);
    p.tiles = q.batch * p.tiles_per_batch;
    if (p.pair) {
        if (t == TG_BF16) pair_numbers<Kind::BF16>(p.block_n, &p.stages, &p.smem, &p.threads, &p.tmem_cols);
        else if (t == TG_FP16) pair_numbers<Kind::FP16>(p.block_n, &p.stages, &p.smem, &p.threads, &p.tmem_cols);
        else if (t == TG_E4M3) pair_numbers<Kind::E4M3>(p.block_n, &p.stages, &p.smem, &p.threads, &p.tmem_cols);
        else pair_numbers<Kind::E5M2>(p.block_n, &p.stages, &p.smem, &p.threads, &p.tmem_cols);
    } else {
        config_numbers_for(t, p.block_n, &p.stages, &p.smem, &p.threads, &p.tmem_cols);
        if (p.producer == 2) p.threads += 4 * 32;  // plain-load producer warps
    }
    // Raster group: M tiles per group.  For 256-row pair tiles, 8 (a window
    // of about 8 x 9.5 tiles per wave of 76 pairs) measured the least DRAM
    // traffic at 8192^3 (1.07 GB per launch, against 1.25 GB for 16 and
    // 1.48 GB for 4); 12 where odd waves walk K downwards (below).
    int64_t g = o->raster_group ? o->raster_group : (p.pair ? 8 : 16);
    if (g > mblocks) g = mblocks;
    p.group = (int)g;
    if (p.pair) {
        // Pairs available, then the split: with fewer tiles than pairs the
        // grid is sized for the tiles' K segments (so every segment gets a
        // pair); otherwise for all pairs, and only the last partial wave can
        // be split.  The kernel applies the same rule to its actual grid.
        const int cl = 2 * p.mc;  // CTAs per cluster
        int64_t pairs_max = sms / cl;
        if (o->max_ctas && pairs_max > o->max_ctas / cl) pairs_max = o->max_ctas / cl;
        if (pairs_max < 1) pairs_max = 1;
        // Tickets: with one pair per cluster and at least a wave of tiles,
        // pairs claim their later tiles in order, so the ones that run ahead
        // take the tail.  Static assignment fixes a pair's tiles, and pairs
        // drift apart by several microseconds over a dozen tiles (8192^3
        // BF16: 7-11 us at the 14th tile); over a few waves the drift is
        // small and the static order measured as fast or faster (4096^3
        // FP16: 89.8 vs 91.7 us), so the planner takes tickets from
        // kTicketMinWaves waves up.  They need the workspace's counter, so
        // not with split_k = 1.
        const bool ticket_ok = p.mc == 1 && o->split_k != 1 && p.tiles >= pairs_max &&
                               (o->schedule == 0 || o->schedule == 4);
        if (o->schedule == 4 && !ticket_ok) return TG_ERR_INVALID_VALUE;
        p.ticket = ticket_ok && (o->schedule == 4 || p.tiles >= kTicketMinWaves * pairs_max);
        // K segments: up to 8 when there are fewer tiles than pairs; with a
        // wave or more, a last wave at most half full is cut into two
        // segments that exchange halves (its tiles then take half a tile's
        // time plus a short fix-up), unless the caller asked for no workspace.
        p.split_max = o->split_k != 0 ? o->split_k : (p.tiles < pairs_max ? kDefaultSplitMax : 2);
        if (p.mc != 1) p.split_max = 1;  // K segments only with one pair per cluster
        int64_t pairs = pairs_max;
        if (p.tiles < pairs_max) {
            int64_t segs = pairs_max / p.tiles;
            if (segs > p.split_max) segs = p.split_max;
            if (segs > nkb / tg::SPLIT_MIN_KBLOCKS) segs = nkb / tg::SPLIT_MIN_KBLOCKS;
            if (segs < 1) segs = 1;
            pairs = p.tiles * segs;
        }
        p.grid = (int)(cl * pairs);
        split_rule(p.tiles, pairs, nkb, p.split_max, sms / 2, &p.split_tiles, &p.split_segs);
        if (o->schedule == 2) {
            // Dynamic: one cluster launched per tile; the hardware starts as
            // many as fit and the running ones take over the rest.
            if (p.mc != 1 || p.tiles > INT32_MAX / 2) return TG_ERR_INVALID_VALUE;
            p.dynamic = true;
            p.ticket = false;
            p.split_max = 1;
            p.split_tiles = 0;
            p.split_segs = 1;
            p.grid = (int)(2 * p.tiles);
        }
        // Many waves of 16-bit tiles: odd waves walk K downwards, so each
        // wave starts on the K blocks the one before read last.  At 8192^3
        // BF16 that cut DRAM reads from 0.99 to 0.87 GB per launch and the
        // sustained launch time by 0.6 %; 4096^3 (static, 3.4 waves) and the
        // 8-bit kinds (twice the bytes per second through L2) did not gain.
        p.k_snake = p.ticket && elem_bytes(t) == 2;
        // With the alternating K order a wave reuses more of the A rows the
        // one before read, and a taller window pays: at 8192^3 DRAM reads of
        // 0.80 GB per launch for 12 M tiles per group, 0.89 GB for 8, 0.85 GB
        // for 16; 200 back-to-back launches 620.6 vs 624.6 us for 8.
        if (p.k_snake && !o->raster_group) p.group = (int)(mblocks < 12 ? mblocks : 12);
    } else {
        if (o->schedule == 2) return TG_ERR_INVALID_VALUE;  // needs CTA-pair tiles
        int64_t grid = p.tiles < cap ? p.tiles : cap;
        if (p.stream_k) {
            // Every CTA up to the cap, at least kStreamKMinBlocks K blocks each.
            grid = p.tiles * nkb / kStreamKMinBlocks;
            if (grid > cap) grid = cap;
        }
        p.grid = (int)(grid < 1 ? 1 : grid);
        // One wave of whole tiles: each tile starts its K loop at its own
        // offset (rotated order).  In step, every CTA reads the same K
        // offset of rows about a megabyte apart at the same time, and on
        // some boxes of the pool that ran 9-11 % slower at 16384 x 64 x 4096
        // (36.5 vs 33.3 us per launch; others saw no difference).  Only where
        // an operand that several tiles share stays in L2 anyway (one N block
        // or a small A-role operand, one M block or a small B-role operand),
        // since the rotated tiles no longer read it together.
        const int64_t e_in = elem_bytes(t);
        const bool a_ok = nblocks == 1 || p.mk * K * e_in <= kRotateSharedBytes;
        const bool b_ok = mblocks == 1 || p.nk * K * e_in <= kRotateSharedBytes;
        p.k_rotate = !p.stream_k && p.tiles <= p.grid && o->schedule != 1 && a_ok && b_ok &&
                     nkb >= kRotateMinBlocks;
    }
    // Swapped roles store each thread's 32 consecutive columns as 16-byte
    // vectors when every row of every batch entry starts 16-byte aligned.
    const int eo = out_bytes(q.out_fmt);
    p.vector_store = p.swap && ((uintptr_t)q.D % 16 == 0) && ((q.ldc * eo) % 16 == 0) &&
                     (q.batch <= 1 || (q.sd * eo) % 16 == 0);
    *plan = p;
    return TG_OK;
}

// ------------------------------------------------------------------ TMA maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// K-major operand: `nb` batch entries (stride `sb` elements apart) of `rows`
// rows of `k` elements, leading stride `ld`; box = 128-byte rows (block_k
// elements) x box_rows x 1 entry, 128-byte swizzle, zero fill outside
// [0,k) x [0,rows).
bool encode_operand(CUtensorMap *map, tg_dtype t, const void *base, int64_t rows, int64_t k,
                    int64_t ld, int64_t nb, int64_t sb, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    if (is_fp4(t)) {  // packed FP4: described as bytes, two elements each
        k = (k + 1) / 2;
        ld /= 2;
        sb /= 2;
        t = TG_E4M3;
    }
    const int e = elem_bytes(t);
    CUtensorMapDataType dt = t == TG_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                             : t == TG_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                             : e == 1       ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                            : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    cuuint64_t dims[3] = {(cuuint64_t)k, (cuuint64_t)rows, (cuuint64_t)nb};
    cuuint64_t strides[2] = {(cuuint64_t)(ld * e), (cuuint64_t)(nb > 1 ? sb * e : ld * e)};
    cuuint32_t box[3] = {(cuuint32_t)(128 / e), (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// A composed epilogue from the caller's op list (checked: count, kinds,
// bias pointers present and float-aligned).
tg_status make_program(const tg_epi_op *ops, int32_t n_ops, tg::EpiProgram *prog) {
    std::memset(prog, 0, sizeof(*prog));
    if (n_ops < 0 || n_ops > tg::EPI_MAX_OPS || (n_ops > 0 && !ops)) return TG_ERR_INVALID_VALUE;
    for (int q = 0; q < n_ops; ++q) {
        const tg_epi_op &o = ops[q];
        if (o.kind < 0 || o.kind >= tg::EPI_KINDS) return TG_ERR_INVALID_VALUE;
        const bool bias = o.kind == TG_EPI_BIAS_ROW || o.kind == TG_EPI_BIAS_COL;
        if (bias && (!o.bias || (uintptr_t)o.bias % 4)) return TG_ERR_INVALID_VALUE;
        prog->op[q].kind = o.kind;
        prog->op[q].a = o.a;
        prog->op[q].b = o.b;
        prog->op[q].bias = bias ? o.bias : nullptr;
    }
    prog->n = n_ops;
    return TG_OK;
}

// With TG_LOG set in the environment, one line per call: the planner's choice.
void log_plan(const char *what, const Problem &q, const Plan &p) {
    if (!std::getenv("TG_LOG")) return;
    std::fprintf(stderr,
                 "%s: M=%lld N=%lld K=%lld batch=%lld -> %s BN=%d mc=%d swap=%d producer=%d "
                 "tiles=%lld grid=%d stages=%d group=%d split=%lldx%d stream_k=%d dynamic=%d "
                 "ticket=%d\n",
                 what, (long long)q.M, (long long)q.N, (long long)q.K, (long long)q.batch,
                 p.pair ? "pair" : "single", p.block_n, p.mc, p.swap ? 1 : 0, p.producer,
                 (long long)p.tiles, p.grid, p.stages, p.group, (long long)p.split_tiles,
                 p.split_segs, p.stream_k ? 1 : 0, p.dynamic ? 1 : 0, p.ticket ? 1 : 0);
}

tg_status run(const Problem &q, tg_epilogue epi, const tg_options *opts, void *stream_ptr,
              const tg::EpiProgram *prog = nullptr) {
    static const tg::EpiProgram kNoOps = {};
    if (!prog) prog = &kNoOps;
    if (epi != TG_EPILOGUE_NONE && epi != TG_EPILOGUE_RELU) return TG_ERR_INVALID_VALUE;
    tg_status st = validate(q, opts);
    if (st != TG_OK) return st;
    if (q.M == 0 || q.N == 0 || q.batch == 0) return TG_OK;
    int dev = 0;
    DeviceState *ds = nullptr;
    st = device_state(&dev, &ds);
    if (st != TG_OK) return st;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    const int relu = epi == TG_EPILOGUE_RELU ? 1 : 0;

    if (q.K == 0) {
        return tg::launch_fill_empty_sum(q.D, q.M, q.N, q.ldc, q.sd, q.batch, q.out_fmt, q.alpha,
                                         relu, *prog, ds->sms, stream) == cudaSuccess
                   ? TG_OK
                   : TG_ERR_CUDA;
    }

    Plan plan;
    st = make_plan(q, opts, ds->sms, &plan);
    if (st != TG_OK) return st;

    tg::LaunchArgs la;
    std::memset(&la, 0, sizeof(la));
    const void *ar = plan.swap ? q.B : q.A;   // A-role operand
    const void *br = plan.swap ? q.A : q.B;   // B-role operand
    const int64_t ldar = plan.swap ? q.ldb : q.lda;
    const int64_t ldbr = plan.swap ? q.lda : q.ldb;
    const int64_t sar = plan.swap ? q.sb : q.sa;
    const int64_t sbr = plan.swap ? q.sa : q.sb;
    const int64_t nba = (q.batch > 1 && sar != 0) ? q.batch : 1;
    const int64_t nbb = (q.batch > 1 && sbr != 0) ? q.batch : 1;
    la.block_n = plan.block_n;
    la.plain_loads = plan.producer == 2;
    la.pair = plan.pair;
    la.mc = plan.mc;
    if (!la.plain_loads) {
        const int b_box = plan.pair ? plan.block_n / 2 : plan.block_n;
        const int a_box = plan.pair && plan.mc == 2 ? tg::BLOCK_M / 2 : tg::BLOCK_M;
        const bool ok = encode_operand(&la.map_a, q.t, ar, plan.mk, q.K, ldar, nba, sar, a_box) &&
                        encode_operand(&la.map_b, q.t, br, plan.nk, q.K, ldbr, nbb, sbr, b_box);
        if (!ok) {
            if (opts && (opts->producer == 1 || opts->cta_pair == 2 || opts->schedule == 2))
                return TG_ERR_INVALID_VALUE;
            la.plain_loads = true;  // shapes the TMA unit cannot describe
            la.pair = false;
            plan.pair = false;
            plan.mc = 1;
            la.mc = 1;
            plan.tiles_per_batch = ceil_div(plan.mk, tg::BLOCK_M) * ceil_div(plan.nk, plan.block_n);
            plan.tiles = q.batch * plan.tiles_per_batch;
            plan.grid = (int)(plan.tiles < ds->sms ? plan.tiles : ds->sms);
            plan.stream_k = false;
        }
    }
    tg::GemmParams &p = la.p;
    p.m = (int32_t)plan.mk;
    p.n = (int32_t)plan.nk;
    p.k = (int32_t)q.K;
    p.num_m_blocks = (int32_t)ceil_div(plan.mk, plan.pair ? 2 * tg::BLOCK_M : tg::BLOCK_M);
    p.num_n_blocks = (int32_t)ceil_div(ceil_div(plan.nk, plan.block_n), plan.mc);
    p.num_k_blocks = (int32_t)ceil_div(q.K, block_k(q.t));
    p.raster_group = plan.group;
    p.relu = relu;
    p.num_tiles = plan.tiles;
    p.tiles_per_batch = plan.tiles_per_batch;
    p.batch = (int32_t)q.batch;
    p.out_fmt = q.out_fmt;
    p.alpha = q.alpha;
    p.vector_store = plan.vector_store ? 1 : 0;
    p.k_rotate = (!la.pair && plan.k_rotate) ? 1 : 0;
    p.k_snake = (la.pair && plan.k_snake) ? 1 : 0;
    p.d = q.D;
    p.d_row_stride = plan.swap ? q.ldc : 1;
    p.d_col_stride = plan.swap ? 1 : q.ldc;
    p.stride_d = q.sd;
    p.a_ptr = ar;
    p.b_ptr = br;
    p.lda = ldar;
    p.ldb = ldbr;
    p.stride_a = q.batch > 1 ? sar : 0;
    p.stride_b = q.batch > 1 ? sbr : 0;
    p.a_bmul = nba > 1 ? 1 : 0;
    p.b_bmul = nbb > 1 ? 1 : 0;
    p.status = ds->status;
    p.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    p.split_max = 1;
    p.l2_hint = (opts && opts->l2_hint == 2) ? 1 : 0;
    p.dynamic = la.pair && plan.dynamic ? 1 : 0;
    p.swap = plan.swap ? 1 : 0;
    p.epi = *prog;
    p.prefetch_k = (opts && opts->prefetch_k > 0) ? opts->prefetch_k : 0;
    if (la.pair && (plan.split_segs > 1 || plan.ticket)) {
        Workspace w;
        st = workspace_for(dev, stream, ds->sms / 2, &w);
        if (st != TG_OK) return st;
        p.split_max = plan.split_segs > 1 ? plan.split_max : 1;
        p.ws_tiles = (int32_t)w.tiles;
        p.ws = w.ws;
        p.flags = w.flags;
        if (plan.ticket) p.ticket = ticket_counter(w.flags, w.tiles);
    }
    if (!la.pair && plan.stream_k) {
        // One 128 x 256 FP32 slot and one flag per CTA: half a pair tile each.
        Workspace w;
        st = workspace_for(dev, stream, ceil_div(plan.grid, 2), &w);
        if (st != TG_OK) return st;
        p.stream_k = 1;
        p.ws = w.ws;
        p.flags = w.flags;
    }
    la.grid = plan.grid;
    log_plan("tg_gemm", q, plan);
    la.device = dev;
    la.stream = stream;

    cudaError_t e;
    if (q.t == TG_BF16) e = tg::launch_bf16(la);
    else if (q.t == TG_FP16) e = tg::launch_fp16(la);
    else if (q.t == TG_E4M3) e = tg::launch_e4m3(la);
    else if (q.t == TG_E5M2) e = tg::launch_e5m2(la);
    else e = tg::launch_tf32(la);
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

// ------------------------------------------------------------------ block-scaled products

// Scale-atom bytes: 128 rows x 4 blocks per 512-byte atom.
int64_t mx_scale_bytes(int64_t rows, int64_t K, tg_dtype t = TG_E4M3) {
    return ceil_div(rows, tg::BLOCK_M) * ceil_div(K, 4 * scale_k(t)) * 512;
}

// Options the block-scaled path honours: tile N (128 or 256), role swap,
// raster group and grid cap; everything else must stay at its default.
bool mx_options_ok(const tg_options *o) {
    if (!o) return true;
    if (o->block_n != 0 && o->block_n != 128 && o->block_n != 256) return false;
    if (o->swap_ab < 0 || o->swap_ab > 2 || o->raster_group < 0 || o->max_ctas < 0) return false;
    if (o->producer < 0 || o->producer > 2) return false;
    if (o->cta_pair < 0 || o->cta_pair == 1 || o->cta_pair > 2) return false;
    if (o->split_k < 0 || o->split_k > 1) return false;
    if (o->l2_hint || o->prefetch_k < -1 || o->prefetch_k > 0) return false;
    if (o->multicast < 0 || o->multicast > 1) return false;
    return o->schedule >= 0 && o->schedule <= 1 && !o->reserved[0];
}

// Scale-atom batch strides (bytes): 0 (one scale set for every entry), or a
// multiple of 16 no smaller than one entry's atoms.
bool mx_scale_stride_ok(int64_t stride, int64_t rows, int64_t K, int64_t batch, tg_dtype t) {
    if (batch <= 1 || stride == 0) return true;
    return stride > 0 && stride % 16 == 0 && stride >= mx_scale_bytes(rows, K, t) &&
           stride < (int64_t)(1ull << 40);
}

// Operands of a block-scaled product the TMA can address (rows and batch
// entries 16-byte aligned, in bytes: packed FP4 holds two elements a byte).
bool mx_tma_legal(const Problem &q) {
    const bool fp4 = is_fp4(q.t);
    const int64_t lda_b = fp4 ? q.lda / 2 : q.lda, ldb_b = fp4 ? q.ldb / 2 : q.ldb;
    const int64_t sa_b = fp4 ? q.sa / 2 : q.sa, sb_b = fp4 ? q.sb / 2 : q.sb;
    return tma_legal(q.A, lda_b, 1) && tma_legal(q.B, ldb_b, 1) &&
           tma_batch_legal(sa_b, 1, q.batch) && tma_batch_legal(sb_b, 1, q.batch);
}

tg_status validate_mx(const Problem &q, const void *sfa, int64_t ssfa, const void *sfb,
                      int64_t ssfb, const tg_options *o) {
    if (q.t != TG_E4M3 && q.t != TG_E5M2 && !is_fp4(q.t)) return TG_ERR_INVALID_VALUE;
    const bool fp4 = is_fp4(q.t);
    Problem qq = q;
    if (fp4) qq.t = TG_E4M3;  // the generic checks, on 1-byte storage
    tg_status st = validate(qq, nullptr);
    if (st != TG_OK) return st;
    if (!mx_options_ok(o)) return TG_ERR_INVALID_VALUE;
    // Packed FP4: rows, batch entries and the reduction hold whole bytes.
    if (fp4 && ((q.lda | q.ldb | q.K) & 1)) return TG_ERR_INVALID_VALUE;
    if (fp4 && q.batch > 1 && ((q.sa | q.sb) & 1)) return TG_ERR_INVALID_VALUE;
    if (!mx_scale_stride_ok(ssfa, q.M, q.K, q.batch, q.t) ||
        !mx_scale_stride_ok(ssfb, q.N, q.K, q.batch, q.t))
        return TG_ERR_INVALID_VALUE;
    if (q.M > 0 && q.N > 0 && q.K > 0 && q.batch > 0) {
        // Operands the TMA cannot address run on the plain-load producer;
        // forcing the TMA producer on them is an error.
        if (o && o->producer == 1 && !mx_tma_legal(q)) return TG_ERR_INVALID_VALUE;
        if (!sfa || !sfb || (uintptr_t)sfa % 16 || (uintptr_t)sfb % 16) return TG_ERR_INVALID_VALUE;
    }
    return TG_OK;
}

// Kernel kind of a block-scaled type.
Kind mx_kind(tg_dtype t) {
    return t == TG_E4M3 ? Kind::E4M3 : t == TG_E5M2 ? Kind::E5M2 : t == TG_E2M1 ? Kind::E2M1
                                                                                : Kind::NVF4;
}

// CTA-pair tiles of 256 x 128 or 256 x 256: the candidate with the smaller
// (waves x cycles per K step), with the same per-step costs as make_plan.
tg_status make_mx_plan(const Problem &q, const tg_options *o, int sms, Plan *plan) {
    static const tg_options kNone = {};
    if (!o) o = &kNone;
    Plan p;
    p.pair = true;
    p.mc = 1;
    p.producer = o->producer ? o->producer : (mx_tma_legal(q) ? 1 : 2);
    if (o->swap_ab == 1) p.swap = false;
    else if (o->swap_ab == 2) p.swap = true;
    else p.swap = (q.M < tg::BLOCK_M) && (q.N >= tg::BLOCK_M) && (q.N >= 2 * q.M);
    p.mk = p.swap ? q.N : q.M;
    p.nk = p.swap ? q.M : q.N;
    int64_t pairs = sms / 2;
    if (o->max_ctas && pairs > o->max_ctas / 2) pairs = o->max_ctas / 2;
    if (pairs < 1) pairs = 1;
    int64_t best = -1;
    for (int bn : {256, 128}) {
        if (o->block_n && o->block_n != bn) continue;
        // The plain-load producer's four extra warps leave the 256-column
        // epilogue short of registers: 128 unless asked for.
        if (!o->block_n && p.producer == 2 && bn == 256) continue;
        const int64_t tiles =
            (q.batch > 1 ? q.batch : 1) * ceil_div(p.mk, 2 * tg::BLOCK_M) * ceil_div(p.nk, bn);
        const int64_t mma = bn / 2, smem = 64 + bn / 4;
        const int64_t est = ceil_div(tiles, pairs) * (mma > smem ? mma : smem);
        if (best < 0 || est < best) {
            best = est;
            p.block_n = bn;
        }
    }
    const int64_t mblocks = ceil_div(p.mk, 2 * tg::BLOCK_M);
    p.tiles_per_batch = mblocks * ceil_div(p.nk, p.block_n);
    p.tiles = (q.batch > 1 ? q.batch : 1) * p.tiles_per_batch;
    tg::mx_config_numbers(mx_kind(q.t), p.block_n, p.producer == 2,
                          &p.stages, &p.smem, &p.threads, &p.tmem_cols);
    int64_t g = o->raster_group ? o->raster_group : 8;
    if (g > mblocks) g = mblocks;
    p.group = (int)g;
    p.grid = (int)(2 * (p.tiles < pairs ? p.tiles : pairs));
    const int eo = out_bytes(q.out_fmt);
    p.vector_store = p.swap && ((uintptr_t)q.D % 16 == 0) && ((q.ldc * eo) % 16 == 0);
    *plan = p;
    return TG_OK;
}

// Scale atoms of an operand with `rows` rows as a 4-D tensor of 32-bit words:
// (128 words = one 512-byte atom, atom column kg, row block rb, batch entry),
// entries `stride` bytes apart (nb == 1: one entry); a box holds `box_kg` x
// `box_rb` atoms of one entry (one K stage of one tile side), and columns or
// row blocks past the end read as zeros.
// With `rep`, a fifth dimension of four with byte stride 0 after the words:
// one box then lands each atom four times over, the copies 512 bytes apart
// (atom-major: the four copies of one atom, then the next row block's).
bool encode_scales(CUtensorMap *map, const void *base, int64_t rows, int64_t K, int64_t atom_k,
                   int64_t nb, int64_t stride, int box_kg, int box_rb, bool rep = false) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int64_t kg = ceil_div(K, atom_k), rb = ceil_div(rows, tg::BLOCK_M);
    const cuuint64_t bstride = (cuuint64_t)(nb > 1 ? stride : rb * kg * 512);
    CUresult r;
    if (rep) {
        cuuint64_t dims[5] = {128, 4, (cuuint64_t)kg, (cuuint64_t)rb, (cuuint64_t)nb};
        cuuint64_t strides[4] = {0, 512, (cuuint64_t)(kg * 512), bstride};
        cuuint32_t box[5] = {128, 4, (cuuint32_t)box_kg, (cuuint32_t)box_rb, 1};
        cuuint32_t estr[5] = {1, 1, 1, 1, 1};
        r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 5, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        cuuint64_t dims[4] = {128, (cuuint64_t)kg, (cuuint64_t)rb, (cuuint64_t)nb};
        cuuint64_t strides[3] = {512, (cuuint64_t)(kg * 512), bstride};
        cuuint32_t box[4] = {128, (cuuint32_t)box_kg, (cuuint32_t)box_rb, 1};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS;
}

// Block-scaled GEMM over `q.batch` entries: scale sets `ssfa` / `ssfb` bytes
// apart (0: shared), then the composed program `prog` (or ReLU alone).
tg_status run_mx(const Problem &q, const void *sfa, int64_t ssfa, const void *sfb, int64_t ssfb,
                 int relu, const tg::EpiProgram &prog, const tg_options *opts, void *stream_ptr) {
    tg_status st = validate_mx(q, sfa, ssfa, sfb, ssfb, opts);
    if (st != TG_OK) return st;
    if (q.M == 0 || q.N == 0 || q.batch == 0) return TG_OK;
    int dev = 0;
    DeviceState *ds = nullptr;
    st = device_state(&dev, &ds);
    if (st != TG_OK) return st;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    if (q.K == 0) {
        return tg::launch_fill_empty_sum(q.D, q.M, q.N, q.ldc, q.sd, q.batch, q.out_fmt, q.alpha,
                                         relu, prog, ds->sms, stream) == cudaSuccess
                   ? TG_OK
                   : TG_ERR_CUDA;
    }
    Plan plan;
    st = make_mx_plan(q, opts, ds->sms, &plan);
    if (st != TG_OK) return st;

    tg::LaunchArgs la;
    std::memset(&la, 0, sizeof(la));
    const void *ar = plan.swap ? q.B : q.A, *br = plan.swap ? q.A : q.B;
    const void *sar = plan.swap ? sfb : sfa, *sbr = plan.swap ? sfa : sfb;
    const int64_t ldar = plan.swap ? q.ldb : q.lda, ldbr = plan.swap ? q.lda : q.ldb;
    const int64_t sa = plan.swap ? q.sb : q.sa, sb = plan.swap ? q.sa : q.sb;
    const int64_t ssa = plan.swap ? ssfb : ssfa, ssb = plan.swap ? ssfa : ssfb;
    const bool many = q.batch > 1;
    const int64_t nba = many && sa ? q.batch : 1, nbb = many && sb ? q.batch : 1;
    const int64_t nsa = many && ssa ? q.batch : 1, nsb = many && ssb ? q.batch : 1;
    const int atom_k = 4 * scale_k(q.t);       // K elements per scale-atom column
    const int kgs = block_k(q.t) / atom_k;      // scale-atom columns per K stage
    // FP8 at BN = 256: the kernel keeps each B atom four times over (its REP
    // layout), loaded through a map with a repeating dimension.
    const bool sfb_rep = !is_fp4(q.t) && plan.block_n == 256;
    la.plain_loads = plan.producer == 2;
    if (!la.plain_loads &&
        (!encode_operand(&la.map_a, q.t, ar, plan.mk, q.K, ldar, nba, sa, tg::BLOCK_M) ||
         !encode_operand(&la.map_b, q.t, br, plan.nk, q.K, ldbr, nbb, sb, plan.block_n / 2) ||
         !encode_scales(&la.map_sfa, sar, plan.mk, q.K, atom_k, nsa, ssa, kgs, 1) ||
         !encode_scales(&la.map_sfb, sbr, plan.nk, q.K, atom_k, nsb, ssb, kgs,
                        plan.block_n / tg::BLOCK_M, sfb_rep)))
        return TG_ERR_INVALID_VALUE;
    la.block_n = plan.block_n;
    la.pair = true;
    la.mc = 1;
    tg::GemmParams &p = la.p;
    p.m = (int32_t)plan.mk;
    p.n = (int32_t)plan.nk;
    p.k = (int32_t)q.K;
    p.num_m_blocks = (int32_t)ceil_div(plan.mk, 2 * tg::BLOCK_M);
    p.num_n_blocks = (int32_t)ceil_div(plan.nk, plan.block_n);
    p.num_k_blocks = (int32_t)ceil_div(q.K, block_k(q.t));
    p.raster_group = plan.group;
    p.relu = relu;
    p.num_tiles = plan.tiles;
    p.tiles_per_batch = plan.tiles_per_batch;
    p.batch = (int32_t)(many ? q.batch : 1);
    p.out_fmt = q.out_fmt;
    p.alpha = q.alpha;
    p.vector_store = plan.vector_store ? 1 : 0;
    p.d = q.D;
    p.d_row_stride = plan.swap ? q.ldc : 1;
    p.d_col_stride = plan.swap ? 1 : q.ldc;
    p.stride_d = many ? q.sd : 0;
    p.a_ptr = ar;
    p.b_ptr = br;
    p.lda = ldar;
    p.ldb = ldbr;
    p.a_bmul = nba > 1 ? 1 : 0;
    p.b_bmul = nbb > 1 ? 1 : 0;
    p.sfa_bmul = nsa > 1 ? 1 : 0;
    p.sfb_bmul = nsb > 1 ? 1 : 0;
    // Plain-load producer: element batch strides (0 when shared) and scale
    // atoms with byte batch strides.
    p.stride_a = nba > 1 ? sa : 0;
    p.stride_b = nbb > 1 ? sb : 0;
    p.sfa_ptr = sar;
    p.sfb_ptr = sbr;
    p.sfa_stride = nsa > 1 ? ssa : 0;
    p.sfb_stride = nsb > 1 ? ssb : 0;
    p.swap = plan.swap ? 1 : 0;
    p.epi = prog;
    p.status = ds->status;
    p.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    p.split_max = 1;
    la.grid = plan.grid;
    log_plan("tg_gemm_mx", q, plan);
    la.device = dev;
    la.stream = stream;
    const cudaError_t e = tg::launch_mx(la, mx_kind(q.t));
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

Problem single(int64_t M, int64_t N, int64_t K, float alpha, const void *A, int64_t lda,
               const void *B, int64_t ldb, void *D, int64_t ldc, tg_dtype t, int out_fmt,
               tg_epilogue epi) {
    return Problem{M, N, K, alpha, A, lda, 0, B, ldb, 0, D, ldc, 0, 1, t, out_fmt,
                   epi == TG_EPILOGUE_RELU ? 1 : 0};
}

}  // namespace

extern "C" {

tg_status tg_gemm(int64_t M, int64_t N, int64_t K, float alpha, const void *A, int64_t lda,
                  const void *B, int64_t ldb, float *D, int64_t ldc, tg_dtype in_dtype,
                  tg_epilogue epilogue, void *stream) {
    return run(single(M, N, K, alpha, A, lda, B, ldb, D, ldc, in_dtype, 0, epilogue), epilogue,
               nullptr, stream);
}

tg_status tg_gemm_ex(int64_t M, int64_t N, int64_t K, float alpha, const void *A, int64_t lda,
                     const void *B, int64_t ldb, float *D, int64_t ldc, tg_dtype in_dtype,
                     tg_epilogue epilogue, const tg_options *opts, void *stream) {
    return run(single(M, N, K, alpha, A, lda, B, ldb, D, ldc, in_dtype, 0, epilogue), epilogue,
               opts, stream);
}

tg_status tg_gemm_batched(int64_t M, int64_t N, int64_t K, float alpha, const void *A,
                          int64_t lda, int64_t stride_a, const void *B, int64_t ldb,
                          int64_t stride_b, void *D, int64_t ldc, int64_t stride_d, int64_t batch,
                          tg_dtype in_dtype, tg_out_dtype out_dtype, tg_epilogue epilogue,
                          const tg_options *opts, void *stream) {
    Problem q{M, N, K, alpha, A, lda, stride_a, B, ldb, stride_b, D, ldc, stride_d, batch,
              in_dtype, (int)out_dtype, epilogue == TG_EPILOGUE_RELU ? 1 : 0};
    return run(q, epilogue, opts, stream);
}

tg_status tg_plan(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
                  int64_t ldb, const float *D, int64_t ldc, tg_dtype in_dtype,
                  const tg_options *opts, int32_t num_sms, tg_plan_info *out) {
    if (!out) return TG_ERR_INVALID_VALUE;
    // NULL operands are planned as 256-byte aligned.
    const void *a = A ? A : reinterpret_cast<const void *>(256);
    const void *b = B ? B : reinterpret_cast<const void *>(256);
    void *d = D ? const_cast<float *>(D) : reinterpret_cast<void *>(256);
    const Problem q = single(M, N, K, 1.0f, a, lda, b, ldb, d, ldc, in_dtype, 0, TG_EPILOGUE_NONE);
    tg_status st = validate(q, opts);
    if (st != TG_OK) return st;
    int sms = num_sms;
    if (sms <= 0) {
        int dev = 0;
        DeviceState *ds = nullptr;
        st = device_state(&dev, &ds);
        if (st != TG_OK) return st;
        sms = ds->sms;
    }
    std::memset(out, 0, sizeof(*out));
    if (M == 0 || N == 0 || K == 0) return TG_OK;  // nothing to tile
    Plan p;
    st = make_plan(q, opts, sms, &p);
    if (st != TG_OK) return st;
    out->block_m = p.pair ? 2 * tg::BLOCK_M : tg::BLOCK_M;
    out->cta_pair = p.pair ? 1 : 0;
    out->split_tiles = (int32_t)p.split_tiles;
    out->split_segs = p.split_segs;
    out->multicast = p.pair ? p.mc : 0;
    out->stream_k = p.stream_k ? 1 : 0;
    out->block_n = p.block_n;
    out->block_k = block_k(in_dtype);
    out->stages = p.stages;
    out->producer = p.producer;
    out->swap_ab = p.swap ? 1 : 0;
    out->raster_group = p.group;
    out->grid = p.grid;
    out->tiles = p.tiles;
    out->threads = p.threads;
    out->smem_bytes = p.smem;
    out->tmem_cols = p.tmem_cols;
    out->vector_store = p.vector_store ? 1 : 0;
    out->schedule = p.dynamic ? 2 : p.stream_k ? 3 : p.ticket ? 4 : 1;
    out->k_rotate = p.k_rotate ? 1 : 0;
    out->k_snake = p.k_snake ? 1 : 0;
    return TG_OK;
}

tg_status tg_plan_describe(int64_t M, int64_t N, int64_t K, tg_dtype in_dtype, int64_t lda,
                           int64_t ldb, int64_t ldc, int32_t num_sms, char *buf, size_t len) {
    if (!buf || len == 0) return TG_ERR_INVALID_VALUE;
    buf[0] = '\0';
    tg_plan_info pi;
    const tg_status st =
        tg_plan(M, N, K, nullptr, lda, nullptr, ldb, nullptr, ldc, in_dtype, nullptr, num_sms, &pi);
    if (st != TG_OK) return st;
    int n;
    if (M == 0 || N == 0 || K == 0) {
        n = std::snprintf(buf, len, "empty");
    } else {
        n = std::snprintf(buf, len,
                          "%s %dx%dx%d stages=%d producer=%s swap=%d grid=%d tiles=%lld raster=%d "
                          "multicast=%d split=%dx%d schedule=%s k_rotate=%d k_snake=%d vector_store=%d "
                          "threads=%d smem=%d tmem=%d",
                          pi.cta_pair ? "pair" : "single", pi.block_m, pi.block_n, pi.block_k,
                          pi.stages, pi.producer == 1 ? "tma" : "plain", pi.swap_ab, pi.grid,
                          (long long)pi.tiles, pi.raster_group, pi.multicast, pi.split_tiles,
                          pi.split_segs,
                          pi.schedule == 2   ? "dynamic"
                          : pi.schedule == 3 ? "stream_k"
                          : pi.schedule == 4 ? "ticket"
                                             : "static",
                          pi.k_rotate, pi.k_snake, pi.vector_store, pi.threads, pi.smem_bytes,
                          pi.tmem_cols);
    }
    return (n >= 0 && (size_t)n < len) ? TG_OK : TG_ERR_INVALID_VALUE;
}

tg_status tg_gemm_epilogue(int64_t M, int64_t N, int64_t K, float alpha, const void *A,
                           int64_t lda, const void *B, int64_t ldb, void *D, int64_t ldc,
                           tg_dtype in_dtype, tg_out_dtype out_dtype, const tg_epi_op *ops,
                           int32_t n_ops, const tg_options *opts, void *stream) {
    tg::EpiProgram prog;
    const tg_status st = make_program(ops, n_ops, &prog);
    if (st != TG_OK) return st;
    const Problem q = single(M, N, K, alpha, A, lda, B, ldb, D, ldc, in_dtype, (int)out_dtype,
                             TG_EPILOGUE_NONE);
    return run(q, TG_EPILOGUE_NONE, opts, stream, &prog);
}

tg_status tg_gemm_mx(int64_t M, int64_t N, int64_t K, float alpha, const void *A, int64_t lda,
                     const void *SFA, const void *B, int64_t ldb, const void *SFB, void *D,
                     int64_t ldc, tg_dtype in_dtype, tg_out_dtype out_dtype, tg_epilogue epilogue,
                     const tg_options *opts, void *stream) {
    if (epilogue != TG_EPILOGUE_NONE && epilogue != TG_EPILOGUE_RELU) return TG_ERR_INVALID_VALUE;
    const Problem q = single(M, N, K, alpha, A, lda, B, ldb, D, ldc, in_dtype, (int)out_dtype,
                             epilogue);
    return run_mx(q, SFA, 0, SFB, 0, epilogue == TG_EPILOGUE_RELU ? 1 : 0, tg::EpiProgram{}, opts,
                  stream);
}

tg_status tg_gemm_mx_batched(int64_t M, int64_t N, int64_t K, float alpha, const void *A,
                             int64_t lda, int64_t stride_a, const void *SFA, int64_t stride_sfa,
                             const void *B, int64_t ldb, int64_t stride_b, const void *SFB,
                             int64_t stride_sfb, void *D, int64_t ldc, int64_t stride_d,
                             int64_t batch, tg_dtype in_dtype, tg_out_dtype out_dtype,
                             const tg_epi_op *ops, int32_t n_ops, const tg_options *opts,
                             void *stream) {
    tg::EpiProgram prog;
    const tg_status st = make_program(ops, n_ops, &prog);
    if (st != TG_OK) return st;
    const Problem q{M, N, K, alpha, A, lda, stride_a, B, ldb, stride_b, D, ldc, stride_d, batch,
                    in_dtype, (int)out_dtype, 0};
    return run_mx(q, SFA, stride_sfa, SFB, stride_sfb, 0, prog, opts, stream);
}

tg_status tg_plan_mx(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                     tg_dtype in_dtype, const tg_options *opts, int32_t num_sms,
                     tg_plan_info *out) {
    if (!out) return TG_ERR_INVALID_VALUE;
    const void *fake = reinterpret_cast<const void *>(256);
    const Problem q = single(M, N, K, 1.0f, fake, lda, fake, ldb, const_cast<void *>(fake), ldc,
                             in_dtype, 0, TG_EPILOGUE_NONE);
    tg_status st = validate_mx(q, fake, 0, fake, 0, opts);
    if (st != TG_OK) return st;
    int sms = num_sms;
    if (sms <= 0) {
        int dev = 0;
        DeviceState *ds = nullptr;
        st = device_state(&dev, &ds);
        if (st != TG_OK) return st;
        sms = ds->sms;
    }
    std::memset(out, 0, sizeof(*out));
    if (M == 0 || N == 0 || K == 0) return TG_OK;
    Plan p;
    st = make_mx_plan(q, opts, sms, &p);
    if (st != TG_OK) return st;
    out->block_m = 2 * tg::BLOCK_M;
    out->block_n = p.block_n;
    out->block_k = block_k(in_dtype);
    out->stages = p.stages;
    out->producer = p.producer;
    out->swap_ab = p.swap ? 1 : 0;
    out->raster_group = p.group;
    out->grid = p.grid;
    out->tiles = p.tiles;
    out->threads = p.threads;
    out->smem_bytes = p.smem;
    out->tmem_cols = p.tmem_cols;
    out->vector_store = p.vector_store ? 1 : 0;
    out->cta_pair = 1;
    out->split_segs = 1;
    out->multicast = 1;
    out->schedule = 1;
    return TG_OK;
}

int64_t tg_mx_scale_bytes(int64_t rows, int64_t K) {
    return tg_bs_scale_bytes(rows, K, TG_E4M3);
}

tg_status tg_mx_pack_scales(int64_t rows, int64_t K, const uint8_t *src, int64_t ld_src,
                            uint8_t *dst, void *stream) {
    return tg_bs_pack_scales(rows, K, TG_E4M3, src, ld_src, dst, stream);
}

int64_t tg_bs_scale_bytes(int64_t rows, int64_t K, tg_dtype in_dtype) {
    if (rows < 0 || K < 0) return -1;
    if (in_dtype != TG_E4M3 && in_dtype != TG_E5M2 && !is_fp4(in_dtype)) return -1;
    return mx_scale_bytes(rows, K, in_dtype);
}

tg_status tg_bs_pack_scales(int64_t rows, int64_t K, tg_dtype in_dtype, const uint8_t *src,
                            int64_t ld_src, uint8_t *dst, void *stream) {
    if (in_dtype != TG_E4M3 && in_dtype != TG_E5M2 && !is_fp4(in_dtype))
        return TG_ERR_INVALID_VALUE;
    const int64_t kblocks = ceil_div(K, scale_k(in_dtype));
    if (rows < 0 || K < 0 || ld_src < (kblocks > 1 ? kblocks : 1)) return TG_ERR_INVALID_VALUE;
    const int64_t total = mx_scale_bytes(rows, K, in_dtype);
    if (total == 0) return TG_OK;
    if (!src || !dst) return TG_ERR_INVALID_VALUE;
    int dev = 0;
    DeviceState *ds = nullptr;
    tg_status st = device_state(&dev, &ds);
    if (st != TG_OK) return st;
    int64_t blocks = ceil_div(total, 256);
    const int64_t cap = (int64_t)ds->sms * 8;
    if (blocks > cap) blocks = cap;
    tg::tg_mx_pack_scales_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        src, rows, kblocks, ld_src, ceil_div(kblocks, 4), total, dst);
    return cudaGetLastError() == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

const char *tg_status_string(tg_status s) {
    switch (s) {
    case TG_OK: return "TG_OK";
    case TG_ERR_INVALID_VALUE: return "TG_ERR_INVALID_VALUE";
    case TG_ERR_UNSUPPORTED: return "TG_ERR_UNSUPPORTED";
    case TG_ERR_CUDA: return "TG_ERR_CUDA";
    case TG_ERR_DEVICE_TIMEOUT: return "TG_ERR_DEVICE_TIMEOUT";
    default: return "TG_ERR_UNKNOWN";
    }
}

tg_status tg_check_device_status(void *stream, int32_t *where) {
    int dev = 0;
    DeviceState *ds = nullptr;
    tg_status st = device_state(&dev, &ds);
    if (st != TG_OK) return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return TG_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, ds->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return TG_ERR_CUDA;
    if (word == 0) return TG_OK;
    if (cudaMemset(ds->status, 0, sizeof(uint32_t)) != cudaSuccess) return TG_ERR_CUDA;
    if (reset_workspace_flags(dev) != TG_OK) return TG_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return TG_ERR_CUDA;
    if (where) *where = (int32_t)word;
    return TG_ERR_DEVICE_TIMEOUT;
}

tg_status tg_set_wait_limit_ns(uint64_t ns) {
    g_wait_limit_ns.store(ns ? ns : kDefaultWaitLimitNs, std::memory_order_relaxed);
    return TG_OK;
}

tg_status tg_selftest_wait_timeout(uint64_t limit_ns, void *stream) {
    if (limit_ns == 0 || limit_ns > 1000000000ull) return TG_ERR_INVALID_VALUE;
    int dev = 0;
    DeviceState *ds = nullptr;
    tg_status st = device_state(&dev, &ds);
    if (st != TG_OK) return st;
    tg::tg_selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(ds->status,
                                                                                 limit_ns);
    return cudaGetLastError() == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

int32_t tg_version(void) { return kVersion; }

}  // extern "C"
