// Persistent, warp-specialised tcgen05 GEMM with a fused alpha/ReLU epilogue.
//
// Computes, in the kernel's "role space", Dk(r, c) = epi(alpha * sum_k Ak(r,k) * Bk(c,k))
// where Ak is the A-role operand (rows r, K-contiguous) and Bk the B-role
// operand (rows c, K-contiguous).  The host either maps A -> Ak, B -> Bk and
// stores Dk(r,c) at D[r + c*ldc] (the natural orientation), or swaps the
// roles (Ak = B's storage, Bk = A's storage) and stores Dk(r,c) at
// D[r*ldc + c]; both operands are K-major, so the swap costs nothing.
//
// Roles per CTA (one CTA per SM, persistent over output tiles):
//   warp 0      producer: one thread issues TMA loads (3-D maps: K, rows,
//               batch entry) into an S-stage ring guarded by full/empty
//               mbarriers ("Walk through GEMM" sections 3-4: copy a K stage,
//               consume, then release it; here the release is the tensor
//               core's own completion signal).
//   warp 1      tensor-memory allocator and MMA issuer: one thread issues
//               tcgen05.mma (128 x BN x 16 for 16-bit kinds, x8 for TF32, x32
//               for 8-bit floats) into one of two TMEM accumulators, FP32
//               ("Matrix Multiplication" step 3: the accumulator is wider than
//               the inputs).
//   warps 2-9   epilogue (warps 2-5 for TF32): tcgen05.ld TMEM -> registers,
//               y = alpha*x, then the max with zero when ReLU is on ("Walk
//               through GEMM" section 5), bounds-checked stores of the
//               rows/columns inside the problem ("Matrix Multiplication",
//               ragged sizes: the overhang is not stored).  A warp reads the
//               TMEM lane quarter warp % 4; with 8 warps each quarter has two,
//               one per half of the columns.  Two accumulators let tile t's
//               epilogue overlap tile t+1's main loop.
//   warps 6-13  (TF32 only) narrow each landed FP32 stage in place to TF32
//               (round to nearest, ties away from zero) before the MMA reads it
//               ("Matrix Multiplication" step 4: convert the operand tiles to
//               TFloat32, keep the accumulator FP32).
//   last 4      (plain-load variant only) the producer: bounds-checked loads
//               that write the TMA's swizzled layout, for strides or bases the
//               TMA cannot address.
// Out-of-range K columns of A and rows of B are read as zeros (TMA
// out-of-bounds fill, or the plain loader's bounds check), which adds nothing
// to the sums ("Matrix Multiplication", ragged sizes: zero padding).
//
// Every wait is bounded in time.  A wait that runs out records a code in the
// per-device status word, raises a CTA-wide abort flag that makes every other
// role leave its loop, drains the copies and MMAs this CTA still has in
// flight (with a bounded wait), frees tensor memory and returns.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include "tg_ptx.cuh"

namespace tg {

enum class Kind : int { BF16 = 0, FP16 = 1, TF32 = 2, E4M3 = 3, E5M2 = 4, E2M1 = 5, NVF4 = 6 };

// Tensor-core instruction family of a kind.
enum class MmaKind : int { F16, TF32, F8, F4 };

template <Kind KD>
struct KindTraits;
template <>
struct KindTraits<Kind::BF16> {
    static constexpr int elem_bytes = 2, block_k = 64, umma_k = 16;
    static constexpr uint32_t fmt = 1;  // instruction-descriptor operand format: BF16
    static constexpr MmaKind mma = MmaKind::F16;
};
template <>
struct KindTraits<Kind::FP16> {
    static constexpr int elem_bytes = 2, block_k = 64, umma_k = 16;
    static constexpr uint32_t fmt = 0;  // F16
    static constexpr MmaKind mma = MmaKind::F16;
};
template <>
struct KindTraits<Kind::TF32> {
    static constexpr int elem_bytes = 4, block_k = 32, umma_k = 8;
    static constexpr uint32_t fmt = 2;  // TF32
    static constexpr MmaKind mma = MmaKind::TF32;
};
// 8-bit floats: one 128-byte swizzle row holds 128 elements; one MMA takes
// 32 of them (32 bytes of K, the same byte step as the 16-bit kinds).
template <>
struct KindTraits<Kind::E4M3> {
    static constexpr int elem_bytes = 1, block_k = 128, umma_k = 32;
    static constexpr uint32_t fmt = 0;  // E4M3 in the f8f6f4 format field
    static constexpr MmaKind mma = MmaKind::F8;
};
template <>
struct KindTraits<Kind::E5M2> {
    static constexpr int elem_bytes = 1, block_k = 128, umma_k = 32;
    static constexpr uint32_t fmt = 1;  // E5M2
    static constexpr MmaKind mma = MmaKind::F8;
};
// Packed 4-bit floats (block-scaled kernel only): two per byte, so one
// 128-byte row holds 256 elements and one MMA (kind::mxf4) takes 64 -- again
// 32 bytes of K.  elem_bytes is not defined for this kind.
template <>
struct KindTraits<Kind::E2M1> {
    static constexpr int block_k = 256, umma_k = 64;
    static constexpr uint32_t fmt = 1;  // E2M1 in the mxf4 format field
    static constexpr MmaKind mma = MmaKind::F4;
};
// The same packed E2M1 operands with NVFP4 scaling (one unsigned-E4M3 scale
// per 16 K elements; kind::mxf4nvf4).
template <>
struct KindTraits<Kind::NVF4> {
    static constexpr int block_k = 256, umma_k = 64;
    static constexpr uint32_t fmt = 1;  // E2M1 in the mxf4nvf4 format field
    static constexpr MmaKind mma = MmaKind::F4;
};

// One tcgen05.mma (single CTA) of the kind's family.
template <Kind KD>
__device__ __forceinline__ void mma_kind(uint32_t d_tmem, uint64_t ad, uint64_t bd, uint32_t idesc,
                                         uint32_t accumulate) {
    if constexpr (KindTraits<KD>::mma == MmaKind::TF32) mma_tf32(d_tmem, ad, bd, idesc, accumulate);
    else if constexpr (KindTraits<KD>::mma == MmaKind::F8) mma_f8(d_tmem, ad, bd, idesc, accumulate);
    else mma_f16(d_tmem, ad, bd, idesc, accumulate);
}

// One tcgen05.mma of a CTA pair (16-bit and 8-bit kinds).
template <Kind KD>
__device__ __forceinline__ void mma_kind_pair(uint32_t d_tmem, uint64_t ad, uint64_t bd,
                                              uint32_t idesc, uint32_t accumulate) {
    static_assert(KindTraits<KD>::mma != MmaKind::TF32, "no TF32 pair tiles");
    if constexpr (KindTraits<KD>::mma == MmaKind::F8) mma_f8_pair(d_tmem, ad, bd, idesc, accumulate);
    else mma_f16_pair(d_tmem, ad, bd, idesc, accumulate);
}

// Codes written to the status word when a bounded wait runs out.
enum WaitSite : uint32_t {
    SITE_FULL = 1,
    SITE_EMPTY = 2,
    SITE_ACC_FULL = 3,
    SITE_ACC_EMPTY = 4,
    SITE_CONVERTED = 5,
    SITE_DRAIN = 6,
    SITE_SELFTEST = 7,
    SITE_SCHED = 10,
    SITE_PARTIAL = 8,
};

// Composed pointwise epilogue: after y = alpha * acc (and the ReLU flag),
// ops[0..n) apply in order to each output value, on the thread that owns it.
enum EpiKind : int32_t {
    EPI_SCALE = 0,      // y = a * y
    EPI_ADD = 1,        // y = y + a
    EPI_RELU = 2,       // y = max(y, 0): NaN stays, -0 becomes +0
    EPI_LEAKY = 3,      // y > 0 ? y : a * y (NaN stays)
    EPI_CLAMP = 4,      // min(max(y, a), b) (NaN stays)
    EPI_SIGMOID = 5,    // 1 / (1 + exp(-y))
    EPI_SILU = 6,       // y / (1 + exp(-y))
    EPI_GELU_TANH = 7,  // y/2 (1 + tanh(sqrt(2/pi) (y + 0.044715 y^3)))
    EPI_BIAS_ROW = 8,   // y + bias[i]
    EPI_BIAS_COL = 9,   // y + bias[j]
    EPI_KINDS = 10,
};
constexpr int EPI_MAX_OPS = 8;
struct EpiOp {
    int32_t kind;
    float a, b;
    const float *bias;  // BIAS_ROW: M values, BIAS_COL: N values (logical rows / columns)
};
struct EpiProgram {
    int32_t n;
    EpiOp op[EPI_MAX_OPS];
};

struct GemmParams {
    int32_t m, n, k;                // role-space problem: rows, cols, reduction
    int32_t num_m_blocks, num_n_blocks, num_k_blocks;
    int32_t raster_group;           // M tiles per raster group
    int32_t relu;
    int64_t num_tiles;
    float alpha;
    int32_t vector_store;           // 1: cols contiguous in D and 16-byte aligned
    void *d;                        // output, element type by out_fmt
    int64_t d_row_stride;           // D element stride between role-space rows
    int64_t d_col_stride;           // D element stride between role-space cols
    const void *a_ptr;              // plain-load producer only
    const void *b_ptr;
    int64_t lda, ldb;               // role-space leading strides (elements)
    uint32_t *status;               // per-device status word
    uint64_t wait_limit_ns;
    // Split-K tail (CTA-pair kernel only): at most `split_max` K segments per
    // tail tile (1 = off); partial tiles go to `ws` (room for `ws_tiles`
    // 256 x 256 pair tiles), with one ready flag per partial half in `flags`.
    int32_t split_max;
    int32_t ws_tiles;
    float *ws;
    uint32_t *flags;
    // L2 policy of the operand loads (CTA-pair kernel): 0 default; 1 A-role
    // rows evict-last (they are reused by every wave of a raster group).
    int32_t l2_hint;
    // Single-CTA TMA producer: every 4 K blocks, prefetch the A-role box of
    // the 4 K blocks `prefetch_k` ahead into L2 in one burst (0 = off), so
    // DRAM sees 512 contiguous bytes of each row at once.
    int32_t prefetch_k;
    // Batches: `batch` independent problems of the same shape.  Tile t is
    // batch entry t / tiles_per_batch.  Operand batch strides are in
    // role-space elements (plain loads); the TMA maps carry them as their
    // third dimension, addressed as b * a_bmul (0: one operand for all).
    int32_t batch;
    int32_t out_fmt;                // 0 FP32, 1 BF16, 2 FP16 output
    int64_t tiles_per_batch;
    int64_t stride_a, stride_b;     // elements between batch entries (role space)
    int64_t stride_d;               // output elements between batch entries
    int32_t a_bmul, b_bmul;
    int32_t sfa_bmul, sfb_bmul;     // block-scaled kernel: scale-atom batch multipliers
    // Block-scaled kernel with the plain-load producer: the role-space scale
    // atoms and their batch strides in bytes (0: one set for every entry).
    const void *sfa_ptr, *sfb_ptr;
    int64_t sfa_stride, sfb_stride;
    // CTA-pair kernel: 1 = dynamic schedule (one cluster launched per tile;
    // running clusters take over clusters not yet started).
    int32_t dynamic;
    // CTA-pair kernel, one pair per cluster: when not NULL, each pair takes
    // its first unit statically and claims every later one in order from
    // this counter (a word of the workspace, zero between launches: the
    // launch's last claim puts it back to zero).
    uint32_t *ticket;
    int32_t swap;                   // 1: role-space rows are D's columns (operands swapped)
    // Single-CTA kernel: 1 = stream-K.  Each CTA takes a contiguous share of
    // the num_tiles x num_k_blocks (tile, K block) iterations; a tile cut
    // between CTAs is finished by the CTA holding its first K block, which
    // adds the later CTAs' FP32 partials (workspace slot = CTA index, 128 x
    // 256 floats each; one ready flag per slot).
    int32_t stream_k;
    // Single-CTA kernel, whole-tile units: 1 = tile t walks its K blocks
    // starting at block (t * K_ROTATE_STEP) mod num_k_blocks (wrapping round),
    // so that the CTAs of a wave do not all read the same K offset of their
    // rows at the same time.  The summation order per tile stays fixed.
    int32_t k_rotate;
    // CTA-pair kernel: 1 = tiles of odd waves (tile / pairs odd) walk their K
    // blocks in descending order, so each wave starts on the K blocks the
    // one before touched last (those most likely still in L2).  The order
    // per tile stays fixed.
    int32_t k_snake;
    EpiProgram epi;                 // composed epilogue (n = 0: alpha and ReLU only)
};

constexpr int BLOCK_M = 128;
constexpr int64_t K_ROTATE_STEP = 13;

// The K block a whole-tile unit of tile t loads at its position kb.
__device__ __forceinline__ int rotated_k_block(const GemmParams &p, int64_t t, int k0, int k1,
                                               int kb, int nkb) {
    if (!p.k_rotate || k0 != 0 || k1 != nkb) return kb;
    int kr = kb + (int)((t * K_ROTATE_STEP) % nkb);
    return kr >= nkb ? kr - nkb : kr;
}
constexpr int ROW_BYTES = 128;                   // one K-major smem row: 128 bytes
constexpr int SMEM_LIMIT = 232448;               // max dynamic smem per CTA (227 KB)

template <int BN>
struct StageCount {
    static constexpr int stage_bytes = (BLOCK_M + BN) * ROW_BYTES;
    static constexpr int fit = (SMEM_LIMIT - 2048) / stage_bytes;
    static constexpr int value = fit > 8 ? 8 : fit;
};

template <Kind KD, int BN>
struct Config {
    using T = KindTraits<KD>;
    static constexpr bool TF32 = (KD == Kind::TF32);
    static constexpr int BK = T::block_k;
    static constexpr int STAGES = StageCount<BN>::value;
    static constexpr int A_BYTES = BLOCK_M * ROW_BYTES;
    static constexpr int B_BYTES = BN * ROW_BYTES;
    static constexpr int A_OFF = 0;
    static constexpr int B_OFF = STAGES * A_BYTES;
    static constexpr int BAR_OFF = B_OFF + STAGES * B_BYTES;
    // full[S], empty[S], converted[S], acc_full[2], acc_empty[2], drain
    static constexpr int FULL0 = 0, EMPTY0 = STAGES, CONV0 = 2 * STAGES;
    static constexpr int ACCF0 = 3 * STAGES, ACCE0 = 3 * STAGES + 2, DRAIN = 3 * STAGES + 4;
    static constexpr int NUM_BARS = 3 * STAGES + 5;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int USED_BYTES = MISC_OFF + 16;
    static constexpr int SMEM_BYTES = USED_BYTES + 1024;  // slack for 1024-byte alignment
    static constexpr int TMEM_COLS = 2 * BN;               // two FP32 accumulators
    // Warps: producer, MMA, then epilogue warps (8 for 16-bit kinds: two per
    // tensor-memory lane quarter, each taking half the columns; 4 for TF32,
    // which adds 8 warps that narrow each landed stage in place).
    static constexpr int EPI_WARPS = TF32 ? 4 : 8;
    static constexpr int CONV_WARPS = TF32 ? 8 : 0;  // TF32: narrow each landed stage
    static constexpr int CONV_THREADS = CONV_WARPS * 32;
    static constexpr int NUM_WARPS = 2 + EPI_WARPS + CONV_WARPS;
    // The plain-load producer runs on LOAD_WARPS extra warps after these.
    static constexpr int LOAD_WARPS = 4;
    static constexpr int threads(bool plain) { return (NUM_WARPS + (plain ? LOAD_WARPS : 0)) * 32; }
    static constexpr int NUM_THREADS = NUM_WARPS * 32;
    static constexpr int MMAS_PER_STAGE = BK / T::umma_k;
    // Instruction descriptor: D FP32 (bit 4), A/B formats (bits 7-9, 10-12),
    // both K-major (bits 15, 16 zero), N >> 3 (bits 17-22), M >> 4 (bits 24-28).
    static constexpr uint32_t IDESC = (1u << 4) | (T::fmt << 7) | (T::fmt << 10) |
                                      ((uint32_t)(BN >> 3) << 17) |
                                      ((uint32_t)(BLOCK_M >> 4) << 24);
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory budget");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M = 128");
    static_assert(TMEM_COLS >= 32 && TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0,
                  "tensor-memory allocation is a power of two in [32, 512]");
    static_assert(BK * T::elem_bytes == ROW_BYTES, "one stage row is one 128-byte swizzle row");
};

struct WaitCtl {
    volatile int *abort_flag;
    uint32_t *status;
    uint64_t limit_ns;
};

// Wait for the phase of `bar` with parity `parity`.  Returns false if the CTA
// is aborting or if this wait ran out of time (then it raises the abort flag
// and records `site`).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const WaitCtl &c,
                                           uint32_t site) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*c.abort_flag) return false;
        if (globaltimer_ns() - t0 > c.limit_ns) {
            *c.abort_flag = 1;
            atomicCAS(c.status, 0u, site);
            return false;
        }
    }
}

// Bounded wait that ignores the abort flag (used while draining).
__device__ __forceinline__ bool wait_phase_drain(uint32_t bar, uint32_t parity, const WaitCtl &c) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > c.limit_ns) {
            atomicCAS(c.status, 0u, (uint32_t)SITE_DRAIN);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void tile_coords(int64_t t, const GemmParams &p, int &mb, int &nb) {
    const int64_t per_group = (int64_t)p.raster_group * p.num_n_blocks;
    const int64_t g = t / per_group;
    const int64_t first_m = g * p.raster_group;
    const int64_t left = (int64_t)p.num_m_blocks - first_m;
    const int gsz = (int)(left < p.raster_group ? left : p.raster_group);
    const int64_t r = t - g * per_group;
    mb = (int)(first_m + r % gsz);
    nb = (int)(r / gsz);
}

// Tile t of the whole (batched) problem: batch entry b and its tile (mb, nb).
__device__ __forceinline__ void batch_tile_coords(int64_t t, const GemmParams &p, int &b, int &mb,
                                                  int &nb) {
    b = (int)(t / p.tiles_per_batch);
    tile_coords(t - (int64_t)b * p.tiles_per_batch, p, mb, nb);
}

// First (tile, K block) iteration of CTA c of g under stream-K.
__device__ __forceinline__ int64_t sk_start(int64_t total, int64_t c, int64_t g) {
    return total * c / g;
}

// The single-CTA kernel's work units, the same sequence for every role:
// whole tiles blockIdx.x, blockIdx.x + gridDim.x, ...; or, under stream-K,
// this CTA's share of the iterations cut at tile boundaries.  A unit is tile
// t, K blocks [k0, k1).
struct TileUnits {
    int64_t pos, end, t;
    int32_t k0, k1;
    __device__ __forceinline__ explicit TileUnits(const GemmParams &p) {
        if (p.stream_k) {
            const int64_t total = p.num_tiles * p.num_k_blocks;
            pos = sk_start(total, blockIdx.x, gridDim.x);
            end = sk_start(total, blockIdx.x + 1, gridDim.x);
        } else {
            pos = end = 0;
        }
        t = (int64_t)blockIdx.x - gridDim.x;
        k0 = k1 = 0;
    }
    __device__ __forceinline__ bool next(const GemmParams &p) {
        const int nkb = p.num_k_blocks;
        if (!p.stream_k) {
            t += gridDim.x;
            k0 = 0;
            k1 = nkb;
            return t < p.num_tiles;
        }
        if (pos >= end) return false;
        t = pos / nkb;
        k0 = (int32_t)(pos - t * nkb);
        const int64_t left = end - pos;
        k1 = left < nkb - k0 ? k0 + (int32_t)left : nkb;
        pos += k1 - k0;
        return true;
    }
};

// Stream-K workspace slot of CTA c: 128 rows x 256 columns of FP32, column-major.
constexpr int64_t SK_SLOT_FLOATS = (int64_t)128 * 256;

__device__ __forceinline__ float apply_epilogue(float x, float alpha, int relu) {
    const float y = alpha * x;
    // max(y, 0) when ReLU is on: NaN stays NaN, -0 and negatives give +0.
    return (relu && !(y > 0.0f) && !(y != y)) ? 0.0f : y;
}

// Output formats of D ("Matrix Multiplication", Step 4: keep the FP32
// accumulator and convert on the way out; round to nearest even).
template <int FMT>
struct OutFormat;
template <>
struct OutFormat<0> {
    using T = float;
    static constexpr int PER16 = 4;  // elements per 16-byte vector
    __device__ static T cvt(float y) { return y; }
    __device__ static uint4 pack(const float *y) {
        return make_uint4(__float_as_uint(y[0]), __float_as_uint(y[1]), __float_as_uint(y[2]),
                          __float_as_uint(y[3]));
    }
};
template <>
struct OutFormat<1> {
    using T = unsigned short;
    static constexpr int PER16 = 8;
    __device__ static T cvt(float y) { return __bfloat16_as_ushort(__float2bfloat16_rn(y)); }
    __device__ static uint4 pack(const float *y) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = (uint32_t)cvt(y[2 * i]) | ((uint32_t)cvt(y[2 * i + 1]) << 16);
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <>
struct OutFormat<2> {
    using T = unsigned short;
    static constexpr int PER16 = 8;
    __device__ static T cvt(float y) { return __half_as_ushort(__float2half_rn(y)); }
    __device__ static uint4 pack(const float *y) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = (uint32_t)cvt(y[2 * i]) | ((uint32_t)cvt(y[2 * i + 1]) << 16);
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// One op of a composed epilogue on a value at logical output (i, j).
__device__ __forceinline__ float epi_op(const EpiOp &o, float y, int64_t i, int64_t j) {
    switch (o.kind) {
    case EPI_SCALE: return o.a * y;
    case EPI_ADD: return y + o.a;
    case EPI_RELU: return (!(y > 0.0f) && !(y != y)) ? 0.0f : y;
    case EPI_LEAKY: return (y > 0.0f || y != y) ? y : o.a * y;
    case EPI_CLAMP: return y < o.a ? o.a : (y > o.b ? o.b : y);
    case EPI_SIGMOID: return 1.0f / (1.0f + expf(-y));
    case EPI_SILU: return y / (1.0f + expf(-y));
    case EPI_GELU_TANH: return 0.5f * y * (1.0f + tanhf(0.7978845608f * (y + 0.044715f * y * y * y)));
    case EPI_BIAS_ROW: return y + o.bias[i];
    case EPI_BIAS_COL: return y + o.bias[j];
    default: return y;
    }
}

// The composed ops on one 32-column chunk of role-space row r: op by op
// (the branch is uniform across the warp), columns col0 .. col0 + 31 of which
// only those below p.n are real.  Kept out of line so that the kernels'
// register budget is set by their main loops, not by this path.
static __device__ __noinline__ void epi_program(const GemmParams &p, int32_t r, int32_t col0,
                                                float *y) {
    for (int q = 0; q < p.epi.n; ++q) {
        const EpiOp o = p.epi.op[q];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int32_t c = col0 + j < p.n ? col0 + j : p.n - 1;  // bias reads stay in range
            const int64_t i = p.swap ? c : r, jj = p.swap ? r : c;
            y[j] = epi_op(o, y[j], i, jj);
        }
    }
}

// Stores of one 32-column chunk: value(j) gives the epilogue's result for
// column col0 + j, converted to the output format, bounded by the problem's
// columns.  D is written once and never read back by the kernel, so the
// stores are marked streaming (evict-first) to keep the operands' lines in
// L2.  A chunk that lies wholly inside the problem takes a branch-free path
// that steps a pointer by the column stride.
template <int FMT, class Value>
__device__ __forceinline__ void store_values(const GemmParams &p, typename OutFormat<FMT>::T *drow,
                                             int32_t col0, Value value) {
    using F = OutFormat<FMT>;
    if (col0 + 32 <= p.n) {
        if (p.vector_store) {
            uint4 *dst = reinterpret_cast<uint4 *>(drow + col0);
#pragma unroll
            for (int j = 0; j < 32; j += F::PER16) {
                float y[F::PER16];
#pragma unroll
                for (int e = 0; e < F::PER16; ++e) y[e] = value(j + e);
                __stcs(dst + j / F::PER16, F::pack(y));
            }
        } else {
            const int64_t cs = p.d_col_stride;
            typename F::T *q = drow + (int64_t)col0 * cs;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                __stcs(q, F::cvt(value(j)));
                q += cs;
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (col0 + j < p.n) __stcs(drow + (int64_t)(col0 + j) * p.d_col_stride, F::cvt(value(j)));
        }
    }
}

// Epilogue store of one 32-column chunk of role-space row r: alpha and the
// ReLU flag inline; a composed epilogue stages the chunk's values first.
template <int FMT>
__device__ __forceinline__ void store_chunk(const GemmParams &p, typename OutFormat<FMT>::T *drow,
                                            int32_t r, int32_t col0, const uint32_t (&v)[32]) {
    if (p.epi.n == 0) {
        store_values<FMT>(p, drow, col0, [&](int j) {
            return apply_epilogue(__uint_as_float(v[j]), p.alpha, p.relu);
        });
    } else {
        float y[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) y[j] = apply_epilogue(__uint_as_float(v[j]), p.alpha, p.relu);
        epi_program(p, r, col0, y);
        store_values<FMT>(p, drow, col0, [&](int j) { return y[j]; });
    }
}

// Row r (role space) of batch entry b: store one chunk in the output format.
__device__ __forceinline__ void epilogue_store(const GemmParams &p, int b, int32_t r, int32_t col0,
                                               const uint32_t (&v)[32]) {
    const int64_t off = (int64_t)b * p.stride_d + (int64_t)r * p.d_row_stride;
    if (p.out_fmt == 0) store_chunk<0>(p, static_cast<float *>(p.d) + off, r, col0, v);
    else if (p.out_fmt == 1) store_chunk<1>(p, static_cast<unsigned short *>(p.d) + off, r, col0, v);
    else store_chunk<2>(p, static_cast<unsigned short *>(p.d) + off, r, col0, v);
}

// Narrow one FP32 bit pattern to TF32: round the magnitude to 10 fraction
// bits, ties away from zero; Inf passes through, NaN becomes a quiet NaN whose
// upper fraction bits are set so that it stays NaN without its low 13 bits.
__device__ __forceinline__ uint32_t narrow_tf32(uint32_t u) {
    if ((u & 0x7F800000u) == 0x7F800000u) {
        return (u & 0x007FFFFFu) ? ((u & 0x80000000u) | 0x7FC00000u) : u;
    }
    return (u + 0x1000u) & 0xFFFFE000u;
}

// Plain-load producer: one stage of `rows` x BK elements into the 128-byte
// swizzled K-major layout (16-byte chunk c of row r lands at chunk c ^ (r & 7)).
// Thread t of the NT loader threads takes chunks t, t + NT, ...; it issues
// the loads of up to 8 chunks before storing any of them, so many loads are
// in flight per thread instead of one chunk's worth.
template <int ELEM_BYTES, int ROWS, int NT>
__device__ __forceinline__ void load_stage_plain(uint8_t *dst, const void *src, int64_t ld,
                                                 int32_t row0, int32_t rows_total, int32_t k0,
                                                 int32_t k_total, int lane) {
    constexpr int EPC = 16 / ELEM_BYTES;  // elements per 16-byte chunk
    constexpr int CHUNKS = ROWS * 8;
    constexpr int PER_LANE = CHUNKS / NT;
    constexpr int BATCH_MAX = ELEM_BYTES == 1 ? 4 : 8;  // 16 byte loads per chunk: fewer
    constexpr int BATCH = PER_LANE < BATCH_MAX ? PER_LANE : BATCH_MAX;
    static_assert(PER_LANE % BATCH == 0, "chunks per lane");
#pragma unroll 1
    for (int b0 = 0; b0 < PER_LANE; b0 += BATCH) {
        uint32_t w[BATCH][4];
#pragma unroll
        for (int i = 0; i < BATCH; ++i) {
            const int ch = lane + (b0 + i) * NT;
            const int r = ch >> 3, c = ch & 7;
            const int32_t gr = row0 + r;
            const bool row_in = gr < rows_total;
            if constexpr (ELEM_BYTES == 1) {
                const uint8_t *s = static_cast<const uint8_t *>(src) + (int64_t)gr * ld;
                uint8_t h[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int32_t gk = k0 + c * EPC + e;
                    h[e] = (row_in && gk < k_total) ? s[gk] : (uint8_t)0;
                }
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w[i][e] = (uint32_t)h[4 * e] | ((uint32_t)h[4 * e + 1] << 8) |
                              ((uint32_t)h[4 * e + 2] << 16) | ((uint32_t)h[4 * e + 3] << 24);
            } else if constexpr (ELEM_BYTES == 2) {
                const uint16_t *s = static_cast<const uint16_t *>(src) + (int64_t)gr * ld;
                uint16_t h[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int32_t gk = k0 + c * EPC + e;
                    h[e] = (row_in && gk < k_total) ? s[gk] : (uint16_t)0;
                }
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w[i][e] = (uint32_t)h[2 * e] | ((uint32_t)h[2 * e + 1] << 16);
            } else {
                const uint32_t *s = static_cast<const uint32_t *>(src) + (int64_t)gr * ld;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int32_t gk = k0 + c * EPC + e;
                    w[i][e] = (row_in && gk < k_total) ? s[gk] : 0u;
                }
            }
        }
#pragma unroll
        for (int i = 0; i < BATCH; ++i) {
            const int ch = lane + (b0 + i) * NT;
            const int r = ch >> 3, c = ch & 7;
            uint4 *out = reinterpret_cast<uint4 *>(dst + r * ROW_BYTES + ((c ^ (r & 7)) << 4));
            *out = make_uint4(w[i][0], w[i][1], w[i][2], w[i][3]);
        }
    }
}

template <Kind KD, int BN, bool PLAIN_LOADS>
__global__ void __launch_bounds__(Config<KD, BN>::threads(PLAIN_LOADS), 1)
    tg_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_b, const GemmParams p) {
    using C = Config<KD, BN>;
    constexpr int S = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    auto bar = [&](int i) -> uint32_t { return sbase + C::BAR_OFF + 8 * i; };
    auto a_stage = [&](int s) -> uint32_t { return sbase + C::A_OFF + s * C::A_BYTES; };
    auto b_stage = [&](int s) -> uint32_t { return sbase + C::B_OFF + s * C::B_BYTES; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
    volatile int *fin_ready = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 8);
    const WaitCtl ctl{abort_flag, p.status, p.wait_limit_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar(C::FULL0 + s), PLAIN_LOADS ? C::LOAD_WARPS * 32 : 1);
            mbar_init(bar(C::EMPTY0 + s), 1);
            mbar_init(bar(C::CONV0 + s), C::CONV_THREADS > 0 ? C::CONV_THREADS : 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar(C::ACCF0 + a), 1);
            mbar_init(bar(C::ACCE0 + a), C::EPI_WARPS);
        }
        mbar_init(bar(C::DRAIN), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (!PLAIN_LOADS && threadIdx.x == 0) {
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_b);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Programmatic dependent launch: every role waits for the preceding grid
    // before its first global-memory access; the TMA producer first works
    // out its first tile and claims its first stage, so that its first load
    // leaves right after the wait.
    griddep_launch();
    const uint32_t tmem_base = *tmem_slot;
    const int nkb = p.num_k_blocks;

    if (PLAIN_LOADS && warp >= C::NUM_WARPS) {
        // ------------------------------------------------------ plain-load producer
        griddep_wait();
        constexpr int NT = C::LOAD_WARPS * 32;
        const int ltid = threadIdx.x - C::NUM_WARPS * 32;
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        constexpr int E = C::T::elem_bytes;
        TileUnits un(p);
        while (ok && un.next(p)) {
            int bt, mb, nb;
            batch_tile_coords(un.t, p, bt, mb, nb);
            const uint8_t *a_src = static_cast<const uint8_t *>(p.a_ptr) + (int64_t)bt * p.stride_a * E;
            const uint8_t *b_src = static_cast<const uint8_t *>(p.b_ptr) + (int64_t)bt * p.stride_b * E;
            for (int kb = un.k0; kb < un.k1; ++kb) {
                if (!wait_phase(bar(C::EMPTY0 + s), ph ^ 1, ctl, SITE_EMPTY)) { ok = false; break; }
                const int kr = rotated_k_block(p, un.t, un.k0, un.k1, kb, nkb);
                load_stage_plain<E, BLOCK_M, NT>(smem + C::A_OFF + s * C::A_BYTES, a_src, p.lda,
                                                 mb * BLOCK_M, p.m, kr * C::BK, p.k, ltid);
                load_stage_plain<E, BN, NT>(smem + C::B_OFF + s * C::B_BYTES, b_src, p.ldb,
                                            nb * BN, p.n, kr * C::BK, p.k, ltid);
                fence_proxy_async_smem();
                mbar_arrive(bar(C::FULL0 + s));
                if (++s == S) { s = 0; ph ^= 1; }
            }
        }
    } else if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (PLAIN_LOADS) {
            // (the plain-load producer runs on the loader warps)
        } else if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            bool waited = false;
            TileUnits un(p);
            while (ok && un.next(p)) {
                int bt, mb, nb;
                batch_tile_coords(un.t, p, bt, mb, nb);
                const int32_t ab = bt * p.a_bmul, bb = bt * p.b_bmul;
                if (!waited && p.prefetch_k > 0) {
                    griddep_wait();
                    waited = true;
                }
                if (p.prefetch_k > 0) {
                    for (int j = un.k0; j < un.k0 + p.prefetch_k && j < un.k1; ++j)
                        tma_prefetch_l2_3d(&tmap_a, j * C::BK, mb * BLOCK_M, ab);
                }
                for (int kb = un.k0; kb < un.k1; ++kb) {
                    if (p.prefetch_k > 0 && ((kb - un.k0) & 3) == 0) {
                        for (int j = 0; j < 4; ++j) {
                            const int kp = kb + p.prefetch_k + j;
                            if (kp < un.k1) tma_prefetch_l2_3d(&tmap_a, kp * C::BK, mb * BLOCK_M, ab);
                        }
                    }
                    if (!wait_phase(bar(C::EMPTY0 + s), ph ^ 1, ctl, SITE_EMPTY)) { ok = false; break; }
                    mbar_arrive_expect_tx(bar(C::FULL0 + s), C::A_BYTES + C::B_BYTES);
                    if (!waited) {
                        griddep_wait();
                        waited = true;
                    }
                    const int kr = rotated_k_block(p, un.t, un.k0, un.k1, kb, nkb);
                    tma_load_3d(a_stage(s), &tmap_a, bar(C::FULL0 + s), kr * C::BK, mb * BLOCK_M, ab);
                    tma_load_3d(b_stage(s), &tmap_b, bar(C::FULL0 + s), kr * C::BK, nb * BN, bb);
                    ++issued;
                    if (++s == S) { s = 0; ph ^= 1; }
                }
            }
            if (!ok) {
                // Let every TMA copy already issued land before the CTA exits.
                for (int st = 0; st < S && st < issued; ++st) {
                    const int64_t last = st + (int64_t)S * ((issued - 1 - st) / S);
                    wait_phase_drain(bar(C::FULL0 + st), (uint32_t)((last / S) & 1), ctl);
                }
            }
        }
        // The warp reaches the block-wide barrier below together: the other
        // lanes wait here for the producing lane.
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        griddep_wait();
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t tl = 0;
            bool ok = true;
            const int wait_bar0 = C::TF32 ? C::CONV0 : C::FULL0;
            const uint32_t wait_site = C::TF32 ? SITE_CONVERTED : SITE_FULL;
            TileUnits un(p);
            for (; ok && un.next(p); ++tl) {
                const uint32_t acc = tl & 1, use = tl >> 1;
                if (!wait_phase(bar(C::ACCE0 + acc), (use & 1) ^ 1, ctl, SITE_ACC_EMPTY)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = un.k0; kb < un.k1; ++kb) {
                    if (!wait_phase(bar(wait_bar0 + s), ph, ctl, wait_site)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a0 = a_stage(s), b0 = b_stage(s);
#pragma unroll
                    for (int kk = 0; kk < C::MMAS_PER_STAGE; ++kk) {
                        const uint64_t ad = smem_desc_sw128(a0 + kk * 32);
                        const uint64_t bd = smem_desc_sw128(b0 + kk * 32);
                        const uint32_t accumulate = ((kb - un.k0) | kk) != 0;
                        mma_kind<KD>(d_tmem, ad, bd, C::IDESC, accumulate);
                    }
                    mma_commit(bar(C::EMPTY0 + s));  // stage s is free once these MMAs finish
                    if (++s == S) { s = 0; ph ^= 1; }
                }
                if (!ok) break;
                mma_commit(bar(C::ACCF0 + acc));     // accumulator ready for the epilogue
            }
            if (!ok) {
                mma_commit(bar(C::DRAIN));
                wait_phase_drain(bar(C::DRAIN), 0, ctl);
            }
        }
        __syncwarp();
    } else if (warp < 2 + C::EPI_WARPS) {
        // ------------------------------------------------------ epilogue
        griddep_wait();
        const int q = warp & 3;                       // TMEM lane quarter of this warp
        const int row_in_tile = q * 32 + lane;
        constexpr int COLS = BN / (C::EPI_WARPS / 4);  // columns of this warp
        const int cbase = ((warp - 2) / 4) * COLS;
        const int etid = threadIdx.x - 64;            // 0 .. EPI_WARPS * 32 - 1
        constexpr uint32_t EPI_THREADS = C::EPI_WARPS * 32;
        const int64_t sk_total = p.num_tiles * (int64_t)nkb;
        uint32_t tl = 0;
        TileUnits un(p);
        for (; un.next(p); ++tl) {
            int bt, mb, nb;
            batch_tile_coords(un.t, p, bt, mb, nb);
            const uint32_t acc = tl & 1, use = tl >> 1;
            const bool got = wait_phase(bar(C::ACCF0 + acc), use & 1, ctl, SITE_ACC_FULL);
            // Stream-K units synchronise the epilogue warps on named barriers,
            // so they leave together: if any thread's wait gave up, all stop.
            if (p.stream_k ? named_bar_any(2, EPI_THREADS, !got) : !got) break;
            tc_fence_after();
            const int32_t r = mb * BLOCK_M + row_in_tile;
            const bool row_ok = r < p.m;
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
            if (un.k0 > 0) {
                // Stream-K contributor (the first unit of this CTA's share):
                // raw FP32 partial sums to this CTA's slot, then its flag.
                float *dst = p.ws + (int64_t)blockIdx.x * SK_SLOT_FLOATS;
#pragma unroll 1
                for (int c0 = cbase; c0 < cbase + COLS; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(taddr + c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        __stcg(dst + (int64_t)(c0 + j) * BLOCK_M + row_in_tile, __uint_as_float(v[j]));
                }
                __threadfence();
                named_bar_sync(1, EPI_THREADS);
                if (etid == 0) st_release_gpu_u32(p.flags + blockIdx.x, 1u);
            } else {
                // Owner of the tile.  Under stream-K with the tile cut (k1 <
                // nkb), CTAs blockIdx.x + 1, ... hold its later K blocks:
                // wait (bounded) for their partials, then add them in CTA order.
                const int64_t tile_end = (un.t + 1) * nkb;
                int64_t c_last = blockIdx.x;  // last contributing CTA
                if (un.k1 < nkb) {
                    while (c_last + 1 < gridDim.x &&
                           sk_start(sk_total, c_last + 1, gridDim.x) < tile_end)
                        ++c_last;
                }
                bool ready = true;
                if (c_last > blockIdx.x) {
                    if (etid == 0) {
                        const uint64_t t0 = globaltimer_ns();
                        for (int64_t c = blockIdx.x + 1; c <= c_last && ready; ++c) {
                            while (ld_acquire_gpu_u32(p.flags + c) == 0u) {
                                if (*abort_flag || globaltimer_ns() - t0 > p.wait_limit_ns) {
                                    if (!*abort_flag) {
                                        *abort_flag = 1;
                                        atomicCAS(p.status, 0u, (uint32_t)SITE_PARTIAL);
                                    }
                                    ready = false;
                                    break;
                                }
                            }
                        }
                        *fin_ready = ready ? 1 : 0;
                    }
                    named_bar_sync(1, EPI_THREADS);
                    ready = *fin_ready != 0;
                    if (ready)
                        for (int64_t c = blockIdx.x + 1; c <= c_last; ++c)
                            (void)ld_acquire_gpu_u32(p.flags + c);
                }
#pragma unroll 1
                for (int c0 = cbase; ready && c0 < cbase + COLS; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(taddr + c0, v);
                    tmem_ld_wait();
                    for (int64_t c = blockIdx.x + 1; c <= c_last; ++c) {
                        const float *src =
                            p.ws + c * SK_SLOT_FLOATS + (int64_t)c0 * BLOCK_M + row_in_tile;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            v[j] = __float_as_uint(__uint_as_float(v[j]) +
                                                   __ldcg(src + (int64_t)j * BLOCK_M));
                    }
                    if (row_ok) epilogue_store(p, bt, r, nb * BN + c0, v);
                }
                if (c_last > blockIdx.x) {
                    // Leave the flags at zero for the next launch.
                    named_bar_sync(1, EPI_THREADS);
                    if (etid == 0 && ready)
                        for (int64_t c = blockIdx.x + 1; c <= c_last; ++c) p.flags[c] = 0u;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::ACCE0 + acc));
        }
    } else if constexpr (C::TF32) {
        // ------------------------------------------------------ TF32 narrowing
        griddep_wait();
        constexpr int NT = C::CONV_THREADS;
        constexpr int NA = C::A_BYTES / 16 / NT, NB = C::B_BYTES / 16 / NT;
        static_assert(C::A_BYTES / 16 % NT == 0 && C::B_BYTES / 16 % NT == 0, "stage split");
        const int ct = threadIdx.x - (2 + C::EPI_WARPS) * 32;  // 0 .. NT-1
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        TileUnits un(p);
        while (ok && un.next(p)) {
            for (int kb = un.k0; kb < un.k1; ++kb) {
                if (!wait_phase(bar(C::FULL0 + s), ph, ctl, SITE_FULL)) { ok = false; break; }
                uint4 *a4 = reinterpret_cast<uint4 *>(smem + C::A_OFF + s * C::A_BYTES) + ct;
                uint4 *b4 = reinterpret_cast<uint4 *>(smem + C::B_OFF + s * C::B_BYTES) + ct;
                // All loads of this thread's share first, then narrow and store.
                uint4 xa[NA], xb[NB];
#pragma unroll
                for (int i = 0; i < NA; ++i) xa[i] = a4[i * NT];
#pragma unroll
                for (int i = 0; i < NB; ++i) xb[i] = b4[i * NT];
#pragma unroll
                for (int i = 0; i < NA; ++i)
                    a4[i * NT] = make_uint4(narrow_tf32(xa[i].x), narrow_tf32(xa[i].y),
                                            narrow_tf32(xa[i].z), narrow_tf32(xa[i].w));
#pragma unroll
                for (int i = 0; i < NB; ++i)
                    b4[i * NT] = make_uint4(narrow_tf32(xb[i].x), narrow_tf32(xb[i].y),
                                            narrow_tf32(xb[i].z), narrow_tf32(xb[i].w));
                fence_proxy_async_smem();
                mbar_arrive(bar(C::CONV0 + s));
                if (++s == S) { s = 0; ph ^= 1; }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace tg
