/*
 * tg_gemm: dense GEMM with a fused pointwise epilogue on GB300 (sm_103a).
 *
 *   D = epi(alpha * A * B),  epi = identity or ReLU (max with zero)
 *
 * The operation is the one defined by "Walk through GEMM" (Tylo.jl manual):
 * the introduction (D = alpha * A * B, optionally ReLU in the epilogue) and
 * section 5 "Apply the epilogue and store by ownership" (alpha is applied to
 * the accumulator first, then the max with zero, with no extra kernel).  The
 * operand formats and the FP32 accumulator follow "Matrix Multiplication"
 * (cuTile.jl tutorial), Step 3 "Looping over K" and Step 4 "Using the tensor
 * cores"; ragged sizes follow its section "Sizes that are not a multiple of
 * the tile shape" (out-of-range K reads count as zero, out-of-range outputs
 * are not stored).
 *
 * Storage ("Walk through GEMM", section 2 "Bind runtime global arrays"), all
 * indices zero-based:
 *   A: logical (M, K), K-contiguous:   a(i,k) = A[i*lda + k],  lda >= max(K,1)
 *   B: logical (K, N), K-contiguous:   b(k,j) = B[k + j*ldb],  ldb >= max(K,1)
 *   D: logical (M, N), M-contiguous:   D[i + j*ldc] (float),   ldc >= max(M,1)
 * Element types: TG_BF16 / TG_FP16 operands are 2-byte storage; TG_TF32
 * operands are FP32 storage narrowed in the kernel to TF32 (10 fraction bits,
 * round to nearest, ties away from zero); TG_E4M3 / TG_E5M2 operands are
 * 1-byte 8-bit floats (the OCP FP8 formats: E4M3 with bias 7, no infinities
 * and NaN at S.1111.111; E5M2 with bias 15, IEEE-style infinities and NaNs),
 * both operands of the same type, with alpha as the per-tensor scale
 * ("Matrix Multiplication", "Where to go from here", names FP8 matmuls as the
 * next step; these are its unscaled-block form).  Products accumulate in FP32; D is
 * FP32.  Only D[i + j*ldc] with i < M, j < N is written: stride padding of D
 * is left untouched, and stride padding of A and B is never read.
 *
 * Ownership: every buffer and the stream belong to the caller and are only
 * borrowed for the call ("Walk through GEMM", section 2: views never copy,
 * allocate or make data ready).  A, B and D are device pointers (or memory the
 * device can address); D must not overlap A or B.  The library keeps state of
 * its own: per device a status word and cached attributes, allocated on the
 * first call on the device; and per (device, stream) a workspace of about
 * 20 MB (the partial sums of tiles whose K loop is split across CTAs, by
 * the pair split tail or stream-K, their ready flags, and the counter from
 * which CTA pairs claim tiles under the ticket schedule), allocated on the
 * first call on that stream that splits a tile or claims tiles and kept
 * until the process exits.  Calls on different streams never share a
 * workspace.  That first allocation synchronises the device, so inside a
 * stream capture either make one call of such a shape on the stream
 * beforehand, pass split_k = 1 (tg_gemm_ex), or use tg_gemm_noalloc.
 *
 * Asynchrony: tg_gemm enqueues its work on `stream` (a cudaStream_t passed as
 * void*, NULL for the legacy default stream) and returns without waiting;
 * results are visible after the stream is synchronised.  Calls on one stream
 * run in order; the kernels use no atomics, so repeated calls with the same
 * inputs give bitwise identical D.
 *
 * Errors: arguments are validated on the host before anything is launched.
 * A non-OK status means nothing was enqueued, except TG_ERR_CUDA returned by a
 * failed launch.  Device-side waits have a time limit; a wait that runs out
 * makes the kernel exit early and sets a per-device status word, which
 * tg_check_device_status reads.
 */
#ifndef TG_GEMM_H
#define TG_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TG_OK = 0,
    TG_ERR_INVALID_VALUE = 1,  /* bad dimension, stride, pointer, enum or option */
    TG_ERR_UNSUPPORTED = 2,    /* valid request this build cannot run (e.g. no sm_103 device) */
    TG_ERR_CUDA = 3,           /* a CUDA runtime/driver call failed */
    TG_ERR_DEVICE_TIMEOUT = 4  /* a kernel's bounded wait ran out (see tg_check_device_status) */
} tg_status;

typedef enum {
    TG_BF16 = 0,  /* bfloat16 operands */
    TG_FP16 = 1,  /* IEEE binary16 operands */
    TG_TF32 = 2,  /* FP32 storage, narrowed to TF32 in the kernel */
    TG_E4M3 = 3,  /* 8-bit float, 4 exponent / 3 fraction bits */
    TG_E5M2 = 4,  /* 8-bit float, 5 exponent / 2 fraction bits */
    TG_E2M1 = 5,  /* 4-bit float (2 exponent / 1 fraction bits), two per byte; tg_gemm_mx only */
    TG_NVF4 = 6   /* TG_E2M1 storage with NVFP4 scaling: one unsigned-E4M3 scale per 16 K
                     elements; tg_gemm_mx only */
} tg_dtype;

/* Output element type of tg_gemm_batched ("Matrix Multiplication", Step 4:
 * the accumulator stays FP32 and the result is converted on the way out,
 * rounding to nearest even). */
typedef enum {
    TG_OUT_F32 = 0,
    TG_OUT_BF16 = 1,
    TG_OUT_F16 = 2
} tg_out_dtype;

typedef enum {
    TG_EPILOGUE_NONE = 0,  /* D = alpha * A*B */
    TG_EPILOGUE_RELU = 1   /* D = max(alpha * A*B, 0); NaN stays NaN, -0 becomes +0 */
} tg_epilogue;

/*
 * D = epi(alpha * A * B) on `stream`.
 *
 * M, N, K >= 0.  M == 0 or N == 0: returns TG_OK and launches nothing.
 * K == 0: D = epi(alpha * 0) over the M x N output (the empty sum).
 * Pointers may be NULL only when the matrix they address is empty
 * (A: M*K == 0, B: K*N == 0, D: M*N == 0).  A and B must be aligned to their
 * element size, D to 4 bytes.  Leading strides as in the storage rules above.
 * Strides or base addresses that the tensor-memory-accelerator (TMA) cannot
 * address (not multiples of 16 bytes) are not errors: the planner routes them
 * to a kernel variant whose producer warp loads with plain bounds-checked
 * loads.
 *
 * Returns TG_OK once the work is enqueued; TG_ERR_INVALID_VALUE for bad
 * arguments (nothing enqueued); TG_ERR_UNSUPPORTED when the current device is
 * not a compute capability 10.3 GPU; TG_ERR_CUDA when a CUDA call fails.
 */
tg_status tg_gemm(int64_t M, int64_t N, int64_t K, float alpha,
                  const void *A, int64_t lda,
                  const void *B, int64_t ldb,
                  float *D, int64_t ldc,
                  tg_dtype in_dtype, tg_epilogue epilogue, void *stream);

/*
 * Planner overrides, for tests and tuning.  A zero-initialised struct (or a
 * NULL pointer) means "the planner decides" for every field.
 */
typedef struct {
    int32_t block_n;      /* 0: planner; else 64, 128 or 256 (tile N of one CTA) */
    int32_t producer;     /* 0: planner; 1: TMA loads (must be legal); 2: plain loads */
    int32_t swap_ab;      /* 0: planner; 1: never swap; 2: always swap the A/B roles */
    int32_t raster_group; /* 0: planner; else number of M tiles per raster group (>= 1) */
    int32_t max_ctas;     /* 0: one CTA per SM; else an upper bound on the persistent grid */
    int32_t cta_pair;     /* 0: planner; 1: single-CTA tiles; 2: CTA-pair tiles (not TF32; TMA) */
    int32_t split_k;      /* 0: planner (pair tiles fewer than pairs: split them into up to 8
                             K segments of >= 8 K blocks; a wave or more: a last wave at most
                             half full into 2 segments that exchange halves); 1: never split
                             (nor stream-K, nor tickets: no workspace);
                             n >= 2: split the last, partial wave into at most n segments */
    int32_t l2_hint;      /* 0: planner (default policy); 1: default L2 policy for operand loads;
                             2: A-role rows evict-last (CTA-pair tiles) */
    int32_t prefetch_k;   /* 0: planner; -1: off; n > 0: single-CTA TMA tiles prefetch the A-role
                             rows n K blocks ahead into L2, 4 blocks per burst */
    int32_t multicast;    /* 0: planner; 1: one CTA pair per cluster; 2: two pairs per cluster
                             sharing their A-role rows by TMA multicast (CTA-pair tiles) */
    int32_t schedule;     /* 0: planner (tickets for CTA-pair tiles with one pair per cluster and
                             at least 6 waves of tiles; stream-K for single-CTA tiles fewer
                             than CTAs; else static); 1: static persistent tiles;
                             2: dynamic: one 2-CTA cluster
                             per tile, running clusters take over clusters not yet started
                             (cluster launch control); CTA-pair tiles, no split-K, no multicast;
                             3: stream-K: single-CTA tiles, each CTA a contiguous share of all
                             (tile, K block) iterations, at least 8 K blocks each; a tile cut
                             between CTAs is finished by the one holding its first K block,
                             adding the others' FP32 partials in CTA order (deterministic).
                             Its CTAs (at most one per SM) wait on one another, so they must
                             all fit on the device at once: where the SMs are restricted (an
                             MPS thread limit), pass 1;
                             4: tickets: CTA-pair tiles, one pair per cluster, a persistent
                             grid; each pair takes its first tile statically and claims every
                             later unit in order from a counter in the stream's workspace, so
                             pairs that run ahead take more of the work (needs the workspace:
                             not with split_k = 1) */
    int32_t reserved[1];  /* must be zero */
} tg_options;

/* What the planner chose for one problem (host only; no CUDA call). */
typedef struct {
    int32_t block_m;      /* tile M: 128 (single CTA) or 256 (CTA pair) */
    int32_t block_n;      /* tile N */
    int32_t block_k;      /* K elements per pipeline stage: 128 bytes of K (64 for 2-byte
                             types, 32 for TF32, 128 for 8-bit floats) */
    int32_t stages;       /* shared-memory ring depth */
    int32_t producer;     /* 1 TMA, 2 plain loads */
    int32_t swap_ab;      /* 1 if the kernel computes D^T = B^T A^T with the roles swapped */
    int32_t raster_group; /* M tiles per raster group */
    int32_t grid;         /* persistent CTAs launched */
    int64_t tiles;        /* output tiles */
    int32_t threads;      /* threads per CTA */
    int32_t smem_bytes;   /* dynamic shared memory per CTA */
    int32_t tmem_cols;    /* tensor-memory columns per CTA */
    int32_t vector_store; /* 1 if the epilogue stores 16-byte vectors (swapped, aligned D) */
    int32_t cta_pair;     /* 1 if a pair of CTAs (a 2-CTA cluster) computes each tile */
    int32_t split_tiles;  /* tiles of the last wave computed as K segments (0: none) */
    int32_t split_segs;   /* K segments per such tile (1: none) */
    int32_t multicast;    /* CTA pairs per cluster sharing A rows (1 or 2; 0 for single-CTA) */
    int32_t stream_k;     /* 1 if single-CTA tiles run as stream-K (each CTA a contiguous share
                             of all (tile, K block) iterations; cut tiles summed in CTA order) */
    int32_t schedule;     /* 1 static, 2 dynamic (cluster launch control), 3 stream-K,
                             4 tickets (see tg_options.schedule) */
    int32_t k_rotate;     /* 1 if each tile walks its K blocks from its own offset (one wave
                             of single-CTA tiles; the order per tile stays fixed) */
    int32_t k_snake;      /* 1 if CTA-pair tiles of odd waves (tile index / pairs odd) walk
                             their K blocks in descending order (16-bit kinds under tickets;
                             the order per tile stays fixed) */
} tg_plan_info;

/* tg_gemm with planner overrides.  Invalid or inapplicable overrides
 * (e.g. TMA forced on a TMA-illegal stride) return TG_ERR_INVALID_VALUE. */
tg_status tg_gemm_ex(int64_t M, int64_t N, int64_t K, float alpha,
                     const void *A, int64_t lda,
                     const void *B, int64_t ldb,
                     float *D, int64_t ldc,
                     tg_dtype in_dtype, tg_epilogue epilogue,
                     const tg_options *opts, void *stream);

/*
 * A batch of independent GEMMs of one shape, with a choice of output type:
 *   for b in [0, batch):  D_b = out(epi(alpha * A_b * B_b))
 * with A_b = A + b*stride_a and B_b = B + b*stride_b (elements of in_dtype)
 * and D_b = D + b*stride_d (elements of out_dtype), each laid out as for
 * tg_gemm ("Matrix Multiplication", "Where to go from here": batched operands
 * along a trailing batch dimension).  stride_a or stride_b may be 0 (one
 * operand shared by every batch entry); outputs may not overlap:
 * stride_d >= ldc*N when batch > 1.  out() rounds the FP32 result to
 * out_dtype (round to nearest even; TG_OUT_F32 stores it as is).
 * D must be aligned to its element size.  batch == 0 launches nothing.
 * Strides that are not multiples of 16 bytes route to plain loads, as in
 * tg_gemm.  Returns as tg_gemm_ex.
 */
tg_status tg_gemm_batched(int64_t M, int64_t N, int64_t K, float alpha,
                          const void *A, int64_t lda, int64_t stride_a,
                          const void *B, int64_t ldb, int64_t stride_b,
                          void *D, int64_t ldc, int64_t stride_d, int64_t batch,
                          tg_dtype in_dtype, tg_out_dtype out_dtype, tg_epilogue epilogue,
                          const tg_options *opts, void *stream);

/*
 * Run the planner only.  `num_sms` > 0 plans for that many SMs without
 * touching CUDA; `num_sms` <= 0 queries the current device.  A, B, D are used
 * only for their alignment (may be NULL when M, N or K is 0; a NULL is taken
 * as 256-byte aligned).  Returns TG_ERR_INVALID_VALUE on the same argument
 * errors as tg_gemm_ex.
 */
tg_status tg_plan(int64_t M, int64_t N, int64_t K,
                  const void *A, int64_t lda, const void *B, int64_t ldb,
                  const float *D, int64_t ldc, tg_dtype in_dtype,
                  const tg_options *opts, int32_t num_sms, tg_plan_info *out);

/*
 * The planner's choice for tg_gemm as one line of text, for logs and tuning
 * (a formatter over tg_plan, host only when num_sms > 0).  The operands are
 * planned as 256-byte aligned.  Writes at most `len` bytes into `buf`,
 * always NUL-terminated when len > 0, e.g.
 *   "pair 256x256x64 stages=7 producer=tma swap=0 grid=152 tiles=1024
 *    raster=12 multicast=1 split=36x2 schedule=ticket k_rotate=0 k_snake=1
 *    vector_store=0 threads=320 smem=230768 tmem=512"   (one line)
 * or "empty" when M, N or K is 0.  Returns TG_OK; TG_ERR_INVALID_VALUE on
 * the argument errors of tg_plan, when buf is NULL or len is 0, or when the
 * text did not fit (buf then holds its truncated, NUL-terminated start).
 */
tg_status tg_plan_describe(int64_t M, int64_t N, int64_t K, tg_dtype in_dtype,
                           int64_t lda, int64_t ldb, int64_t ldc, int32_t num_sms,
                           char *buf, size_t len);

/*
 * Block-scaled (microscaling) FP8 GEMM ("Matrix Multiplication", "Where to
 * go from here": block-scaled FP8 matmuls; the pages fix no format, this is
 * the OCP Microscaling one):
 *   D = out(epi(alpha * s)),  s(i,j) = sum over kb of Xa(i,kb) * Xb(kb,j) *
 *                                      sum_{k in block kb} a(i,k) * b(k,j)
 * where block kb covers k in [32*kb, 32*kb + 32) and each scale is a power of
 * two 2^(e-127) given by an 8-bit code e (e = 255 is NaN).  in_dtype is
 * TG_E4M3, TG_E5M2 or TG_E2M1 (both operands); A, B and D are laid out as for
 * tg_gemm (D of type out_dtype).  TG_NVF4 is the other published FP4 scaling
 * (NVFP4): TG_E2M1 operands, blocks of 16 consecutive K elements, and each
 * scale an unsigned E4M3 code (4 exponent bits with bias 7, 3 fraction bits:
 * (1 + m/8) * 2^(e-7), subnormal m/8 * 2^-6 for e = 0, code 0x7F NaN; codes
 * with the top bit set are not scales and give undefined results) -- the
 * sum above with 16 in place of 32.  A and B whose base, row stride or batch
 * stride (in bytes) is not a multiple of 16 run on a kernel variant whose
 * producer warps load with plain bounds-checked loads (producer 2 in the
 * plan; forcing producer 1 on them is TG_ERR_INVALID_VALUE).  TG_E2M1 (FP4:
 * magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6) is packed two per byte, element 2t
 * in the low nibble of byte t of its row; lda, ldb, K (and batch strides)
 * count elements and must be even.
 *
 * Scales (SFA for the M rows of A, SFB for the N columns of B) are stored as
 * "scale atoms": with R rows and KB = ceil(K/32) blocks (TG_NVF4:
 * ceil(K/16)), atom (rb, kg), for
 * rows [128*rb, 128*rb + 128) and blocks [4*kg, 4*kg + 4), is 512 contiguous
 * bytes at byte offset (rb * ceil(KB/4) + kg) * 512, and the scale of row r,
 * block kb is at byte (r % 32) * 16 + ((r / 32) % 4) * 4 + (kb % 4) of its
 * atom.  The buffer holds tg_mx_scale_bytes(R, K) bytes, 16-byte aligned;
 * entries for rows >= R or blocks >= KB are padding and must not be NaN
 * codes (zero is the usual fill).  tg_mx_pack_scales (32-element blocks) and
 * tg_bs_pack_scales (any block-scaled type) write this layout from row-major
 * scales; tg_mx_scale_bytes / tg_bs_scale_bytes size it.
 *
 * opts may set block_n (128 or 256), swap_ab, raster_group, max_ctas and
 * producer (1 TMA, 2 plain loads); any other field must be 0 (or the value
 * that forces what this path does: cta_pair 2, split_k 1, multicast 1,
 * prefetch_k -1).  Returns as tg_gemm_ex.
 */
tg_status tg_gemm_mx(int64_t M, int64_t N, int64_t K, float alpha,
                     const void *A, int64_t lda, const void *SFA,
                     const void *B, int64_t ldb, const void *SFB,
                     void *D, int64_t ldc,
                     tg_dtype in_dtype, tg_out_dtype out_dtype, tg_epilogue epilogue,
                     const tg_options *opts, void *stream);

/* The tg_gemm_mx planner without launching (num_sms as for tg_plan). */
tg_status tg_plan_mx(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                     tg_dtype in_dtype, const tg_options *opts, int32_t num_sms,
                     tg_plan_info *out);

/* Bytes of the scale-atom buffer for `rows` rows and K (-1 on negative input). */
int64_t tg_mx_scale_bytes(int64_t rows, int64_t K);

/*
 * Rewrite row-major scales (row r, block kb at src[r*ld_src + kb], ld_src >=
 * ceil(K/32)) as scale atoms into dst (tg_mx_scale_bytes(rows, K) bytes),
 * padding with zeros, on `stream`.  Both are device buffers.
 */
tg_status tg_mx_pack_scales(int64_t rows, int64_t K, const uint8_t *src, int64_t ld_src,
                            uint8_t *dst, void *stream);

/* Bytes of the scale-atom buffer of in_dtype (TG_E4M3, TG_E5M2, TG_E2M1: one
 * scale per 32 K; TG_NVF4: per 16) for `rows` rows and K; -1 on negative
 * input or a type without block scales. */
int64_t tg_bs_scale_bytes(int64_t rows, int64_t K, tg_dtype in_dtype);

/* tg_mx_pack_scales for in_dtype's block size: row-major scales (row r,
 * block kb at src[r*ld_src + kb], ld_src >= the block count) into
 * tg_bs_scale_bytes(rows, K, in_dtype) bytes of scale atoms at dst. */
tg_status tg_bs_pack_scales(int64_t rows, int64_t K, tg_dtype in_dtype, const uint8_t *src,
                            int64_t ld_src, uint8_t *dst, void *stream);

/*
 * Composed pointwise epilogue ("Walk through GEMM", section 5: the epilogue
 * is a pointwise map of the accumulator, applied by the thread that owns each
 * value; "Tylo README", worked consumers: composed epilogues):
 *   y = alpha * sum_k a(i,k) b(k,j),  then  y = op_n(... op_1(y)),
 *   D[i + j*ldc] = out(y)
 * with each op one of the kinds below (a, b its float arguments; bias a device
 * array of floats).  Everything else is as tg_gemm_batched with batch = 1
 * (any output type).  At most TG_EPI_MAX_OPS ops; n_ops = 0 gives alpha * AB.
 * Returns TG_ERR_INVALID_VALUE for an unknown kind, a missing or misaligned
 * bias pointer, or n_ops out of range, besides tg_gemm_ex's errors.
 */
#define TG_EPI_MAX_OPS 8
typedef enum {
    TG_EPI_SCALE = 0,      /* y = a * y */
    TG_EPI_ADD = 1,        /* y = y + a */
    TG_EPI_RELU = 2,       /* y = max(y, 0) (NaN stays NaN, -0 becomes +0) */
    TG_EPI_LEAKY_RELU = 3, /* y = y > 0 ? y : a * y (NaN stays) */
    TG_EPI_CLAMP = 4,      /* y = min(max(y, a), b) (NaN stays) */
    TG_EPI_SIGMOID = 5,    /* y = 1 / (1 + exp(-y)) */
    TG_EPI_SILU = 6,       /* y = y / (1 + exp(-y)) */
    TG_EPI_GELU_TANH = 7,  /* y = y/2 * (1 + tanh(sqrt(2/pi) * (y + 0.044715 y^3))) */
    TG_EPI_BIAS_ROW = 8,   /* y = y + bias[i], bias: M floats */
    TG_EPI_BIAS_COL = 9    /* y = y + bias[j], bias: N floats */
} tg_epi_kind;

typedef struct {
    int32_t kind;        /* tg_epi_kind */
    float a, b;          /* arguments (unused ones ignored) */
    const float *bias;   /* TG_EPI_BIAS_ROW / TG_EPI_BIAS_COL only; borrowed, device memory */
} tg_epi_op;

tg_status tg_gemm_epilogue(int64_t M, int64_t N, int64_t K, float alpha,
                           const void *A, int64_t lda, const void *B, int64_t ldb,
                           void *D, int64_t ldc, tg_dtype in_dtype, tg_out_dtype out_dtype,
                           const tg_epi_op *ops, int32_t n_ops,
                           const tg_options *opts, void *stream);

/*
 * Batched block-scaled GEMM with a composed epilogue: for b in [0, batch),
 *   D_b = out(op_n(... op_1(alpha * s_b)))
 * with s_b the block-scaled product of tg_gemm_mx on A_b = A + b*stride_a,
 * B_b = B + b*stride_b (elements; for TG_E2M1 and TG_NVF4 the strides count
 * elements and must be even), scales SFA_b = SFA + b*stride_sfa and SFB_b = SFB +
 * b*stride_sfb (bytes), and D_b = D + b*stride_d (elements of out_dtype),
 * each as in tg_gemm_mx; ops as in tg_gemm_epilogue, the same for every
 * entry (a bias is indexed by the row or column within the entry).  Any of
 * stride_a, stride_b, stride_sfa, stride_sfb may be 0 (shared by every
 * entry); outputs may not overlap: stride_d >= ldc*N when batch > 1.  A
 * nonzero scale stride must be a multiple of 16 and at least the bytes of one
 * entry's atoms (tg_bs_scale_bytes); operand batch strides that are not
 * 16-byte multiples run on the plain-load producer, as in tg_gemm_mx.
 * batch == 0 launches nothing; K == 0 writes out(ops(0)).
 * opts as for tg_gemm_mx.  Returns as tg_gemm_mx and tg_gemm_epilogue.
 */
tg_status tg_gemm_mx_batched(int64_t M, int64_t N, int64_t K, float alpha,
                             const void *A, int64_t lda, int64_t stride_a,
                             const void *SFA, int64_t stride_sfa,
                             const void *B, int64_t ldb, int64_t stride_b,
                             const void *SFB, int64_t stride_sfb,
                             void *D, int64_t ldc, int64_t stride_d, int64_t batch,
                             tg_dtype in_dtype, tg_out_dtype out_dtype,
                             const tg_epi_op *ops, int32_t n_ops,
                             const tg_options *opts, void *stream);

/* Static text for a status code ("TG_OK", ...); never NULL. */
const char *tg_status_string(tg_status status);

/*
 * Synchronise `stream`, then read and clear the current device's status word
 * that kernels set when a bounded wait runs out.  Returns TG_OK if no wait ran
 * out since the last check, TG_ERR_DEVICE_TIMEOUT if one did (then *where, if
 * not NULL, receives a code naming the wait: 1 stage-full, 2 stage-empty,
 * 3 accumulator-full, 4 accumulator-empty, 5 converted-stage, 6 drain,
 * 7 self-test), TG_ERR_CUDA on a CUDA error.
 */
tg_status tg_check_device_status(void *stream, int32_t *where);

/*
 * Set the time limit, in nanoseconds, of every device-side wait of later
 * launches on all devices (default 4e9 ns; 0 restores the default).
 */
tg_status tg_set_wait_limit_ns(uint64_t ns);

/*
 * Failure-detection self-test: launch one CTA whose single thread waits on a
 * shared-memory barrier that nothing ever completes, with a `limit_ns` time
 * limit.  The wait runs out, the kernel records code 7 in the status word and
 * returns normally (no trap, no fault); tg_check_device_status then reports
 * TG_ERR_DEVICE_TIMEOUT.  limit_ns must be in (0, 1e9].
 */
tg_status tg_selftest_wait_timeout(uint64_t limit_ns, void *stream);

/*
 * tg_gemm for callers that cannot allocate device memory.  The pages have no
 * counterpart of this call; it exists for callers whose device memory is
 * all held by their own pool allocator, that must avoid cudaMalloc's
 * implicit synchronisation, or that run inside a stream capture where
 * cudaMalloc is not allowed.
 *
 * Same arguments, results and errors as tg_gemm, and the same kernel and
 * planner.  It calls no cudaMalloc, cudaFree or other allocating routine: the
 * kernel's scratch (its 4-byte status word) lives in a fixed 256-byte,
 * 256-byte-aligned __device__ array inside the library, which every device
 * that loads the library holds until the process exits.  A plan needing more
 * scratch than that returns TG_ERR_UNSUPPORTED before launching anything
 * (no M, N, K does today: the status word does not grow with the problem).
 * It never splits a tile's K loop across CTAs, since the partial sums would
 * need a workspace; its K == 0 case runs tg_gemm's fill kernel.
 *
 * The first call on a device, with that device current, looks up the
 * array's device address (cudaGetSymbolAddress); make that first call before
 * any stream capture.  All calls on a device share the array: each call
 * clears the status word on its own stream first, and calls that overlap on
 * the GPU (concurrent streams) race on it.  A wait that runs out still ends
 * the kernel early, but this call does not report it (tg_check_device_status
 * reads only tg_gemm's word); its waits use the default 4 s limit.
 */
tg_status tg_gemm_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                          const void *A, int64_t lda,
                          const void *B, int64_t ldb,
                          float *D, int64_t ldc,
                          tg_dtype in_dtype, tg_epilogue epilogue, void *stream);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t tg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TG_GEMM_H */
