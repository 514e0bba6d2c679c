// Block-scaled (microscaling) FP8 GEMM on CTA pairs.
//
//   D = epi(alpha * sum_kb Xa(i,kb) Xb(kb,j) sum_{k in kb} a(i,k) b(k,j))
//
// with E4M3 / E5M2 operands and one 8-bit power-of-two scale (2^(e-127)) per
// 32 consecutive K elements of each A row and each B column ("Matrix
// Multiplication", "Where to go from here": block-scaled FP8 matmuls; the
// scale format is the OCP Microscaling one).  The tensor core applies the
// scales itself: tcgen05.mma.kind::mxf8f6f4.block_scale reads them from
// tensor memory next to the accumulator.
//
// Scale storage ("scale atoms"): for an operand with R rows (A: M, B: N) and
// KB = ceil(K/32) scale blocks, the scales are grouped in atoms of 128 rows x
// 4 blocks = 512 contiguous bytes; atom (rb, kg) starts at byte
// (rb * ceil(KB/4) + kg) * 512, and inside it the scale of row r, block kb
// sits at byte (r % 32) * 16 + ((r / 32) % 4) * 4 + kb % 4.  That is the
// order in which one 32-lane x 16-byte tcgen05.cp, repeated over the four
// lane quarters, puts row r's four scales in tensor-memory column r / 32,
// bytes 0-3 (lane r % 32 of every quarter) -- where the block-scaled MMA
// reads them, one byte per 32-wide MMA chosen by the descriptor's scale ID.
//
// One 128-byte K stage holds 128 FP8 elements = 4 scale blocks = one atom
// column, so a stage carries one A atom per CTA and BN/128 B atoms; with
// packed FP4 (E2M1) a stage holds 256 elements = two atom columns, and each
// 64-wide MMA (kind::mxf4, two scales per row) reads bytes (0, 1) or (2, 3).
// NVFP4 (Kind::NVF4: the same packed E2M1 operands, one unsigned-E4M3 scale
// per 16 K elements) keeps the atom layout with 16-element blocks: an atom
// column covers 64 K, a stage four of them, and each 64-wide MMA
// (kind::mxf4nvf4, scale_vec::4X) reads all four bytes of its column's word.
//
// Differences from the CTA-pair kernel of tg_kernel_pair.cuh:
//   - each stage also lands its scale atoms (TMA, 512 bytes each); each CTA
//     loads the A atom of its own 128 rows and all BN/128 B atoms (every
//     CTA's tensor core scales all BN columns);
//   - the MMA thread copies a stage's atoms into that stage's tensor-memory
//     slot (tcgen05.cp) right before the stage's four MMAs; a slot is reused
//     only after the producer has refilled the stage, which waits for those
//     MMAs to finish, so no copy can overwrite scales still being read;
//   - one accumulator (the scale slots take the rest of tensor memory): the
//     epilogue warps load their whole share of the tile into registers,
//     release the accumulator at once, and store from registers while the
//     next tile's MMAs run;
//   - no split-K tail, no multicast clusters.
// With PLAIN = true (operand strides or bases the TMA cannot address), four
// more warps per CTA copy each stage with bounds-checked plain loads (the
// operands into the TMA's swizzled layout, zeros beyond K and beyond the
// rows; the 512-byte scale atoms as they are, zeros past the last atom column
// or row block), and every loader thread of both CTAs arrives on the pair
// leader's stage-full barrier (the peer's remotely, with release semantics at
// cluster scope).
// Every wait is bounded as in the other kernels.
#pragma once

#include <cstdint>
#include "tg_kernel_pair.cuh"

namespace tg {

template <Kind KD, int BN>
struct MxConfig {
    using T = KindTraits<KD>;
    static constexpr bool FP4 = T::mma == MmaKind::F4;   // packed E2M1 operands
    static constexpr bool NV = KD == Kind::NVF4;         // 16-element unsigned-E4M3 scales
    static_assert(T::mma == MmaKind::F8 || FP4, "block scaling covers the 8- and 4-bit floats");
    static_assert(BN == 128 || BN == 256, "tile N: whole 128-row scale atoms");
    static constexpr int BK = T::block_k;                // K elements per stage (128 / 256)
    static constexpr int BK_UNITS = ROW_BYTES;           // the same in tensor-map units (bytes)
    static constexpr int PAIR_M = 2 * BLOCK_M;
    static constexpr int B_ROWS = BN / 2;
    static constexpr int SFB_ATOMS = BN / 128;           // B atoms per atom column
    static constexpr int SCALE_K = NV ? 16 : 32;         // K elements per scale
    static constexpr int ATOM_K = 4 * SCALE_K;           // K elements per atom column
    static constexpr int KGS = BK / ATOM_K;              // atom columns per stage (4 blocks each)
    static constexpr int ATOM_BYTES = 512;
    static constexpr int A_BYTES = BLOCK_M * ROW_BYTES;
    static constexpr int B_BYTES = B_ROWS * ROW_BYTES;
    // FP8 at BN = 256 (one atom column, two B row blocks): each B atom is
    // stored four times over (2 KB: the 32 rows of the atom for each of the
    // four 32-lane quarters), so that one 128-lane tcgen05.cp of 32-byte rows
    // moves both B atoms -- two copies per stage instead of three, and a
    // copy's tensor-pipe time goes by instruction, not by bytes.
    static constexpr bool REP = !FP4 && SFB_ATOMS == 2;
    static constexpr int REP_BYTES = 4 * ATOM_BYTES;     // one atom, four quarters
    static constexpr int SFA_BYTES = KGS * ATOM_BYTES;   // [kg][atom]
    static constexpr int SFB_BYTES =                     // [row block][kg][atom] (x4 if REP)
        KGS * SFB_ATOMS * ATOM_BYTES * (REP ? 4 : 1);
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
    static constexpr int FIT = (SMEM_LIMIT - 2048) / STAGE_BYTES;
    static constexpr int STAGES = FIT > 8 ? 8 : FIT;
    // Operand tiles (1024-byte aligned for the 128-byte swizzle) after the
    // scales when REP, so that nothing a 4 KB scale copy reads lies past
    // the end of shared memory; before them otherwise.
    static constexpr int SCALE_REGION = STAGES * (SFA_BYTES + SFB_BYTES);
    static constexpr int A_OFF = REP ? (SCALE_REGION + 1023) / 1024 * 1024 : 0;
    static constexpr int B_OFF = A_OFF + STAGES * A_BYTES;
    static constexpr int SFB_OFF = REP ? 0 : B_OFF + STAGES * B_BYTES;
    static constexpr int SFA_OFF = SFB_OFF + STAGES * SFB_BYTES;
    static constexpr int BAR_OFF = REP ? B_OFF + STAGES * B_BYTES : SFA_OFF + STAGES * SFA_BYTES;
    static constexpr int FULL0 = 0, EMPTY0 = STAGES;
    static constexpr int ACCF = 2 * STAGES, ACCE = 2 * STAGES + 1, DRAIN = 2 * STAGES + 2;
    static constexpr int NUM_BARS = 2 * STAGES + 3;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;
    // Tensor memory: the accumulator in columns [0, BN); then one scale slot
    // per stage: A atoms at +4*kg .. +4*kg+3, B atoms from SFB_COL, atom
    // column kg at SFB_COL + 4*SFB_ATOMS*kg (+4 per row block).
    static constexpr int SFB_COL = 4 * KGS > 8 ? 4 * KGS : 8;
    static constexpr int SFB_COLS = 4 * SFB_ATOMS * KGS;
    static constexpr int SLOT_COLS = (SFB_COL + SFB_COLS + 15) / 16 * 16;
    static constexpr int SF_COL0 = BN;
    static constexpr int USED_COLS = BN + STAGES * SLOT_COLS;
    static constexpr int TMEM_COLS = USED_COLS <= 256 ? 256 : 512;
    static constexpr int EPI_WARPS = 8;
    static constexpr int NUM_WARPS = 2 + EPI_WARPS;
    static constexpr int NUM_THREADS = NUM_WARPS * 32;
    static constexpr int LOAD_WARPS = 4;  // plain-load producer, after the others
    static constexpr int threads(bool plain) { return (NUM_WARPS + (plain ? LOAD_WARPS : 0)) * 32; }
    static constexpr int MMAS_PER_STAGE = BK / T::umma_k;  // 4: one per scale block
    static constexpr int COLS = BN / 2;                      // columns per epilogue warp
    // Block-scaled instruction descriptor: B scale ID (bits 4-5, per MMA),
    // A/B formats (7-9, 10-12), K-major operands (15, 16 zero), N >> 3
    // (17-22), scale type (bit 23: 1 = 8-bit exponent, 0 = unsigned E4M3),
    // M >> 4 (24-28), A scale ID (29-30, per MMA).
    static constexpr uint32_t IDESC = (T::fmt << 7) | (T::fmt << 10) |
                                      ((uint32_t)(BN >> 3) << 17) | ((NV ? 0u : 1u) << 23) |
                                      ((uint32_t)(PAIR_M >> 4) << 24);
    // MMA kk of a stage: the atom column holding its scales, and the byte of
    // each 32-bit scale word it starts at (its K offset inside the column, in
    // scale blocks): FP8 byte kk of column 0; MX FP4 bytes 0 / 2 of column
    // kk / 2; NVFP4 the whole word of column kk.
    __host__ __device__ static constexpr int atom_col(int kk) { return kk * T::umma_k / ATOM_K; }
    __host__ __device__ static constexpr uint32_t scale_id(int kk) {
        return (uint32_t)((kk * T::umma_k) % ATOM_K / SCALE_K);
    }
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory budget");
    static_assert(A_OFF % 1024 == 0 && B_OFF % 1024 == 0, "swizzled operand tiles");
    static_assert(!REP || KGS == 1, "replicated B atoms: one atom column per stage");
    static_assert(STAGES >= 4, "pipeline depth");
    static_assert(USED_COLS <= 512, "tensor memory");
    static_assert(4 * KGS <= SFB_COL, "A atoms fit below the B atoms");
};

// Per-MMA descriptor: the same scale ID for both operands.
__device__ __forceinline__ uint32_t mx_idesc(uint32_t base, uint32_t id) {
    return base | (id << 4) | (id << 29);
}

// Plain-load copy of `count` 512-byte scale atoms, atom i taken from atom
// column kg0 + (i % kgs) of row block rb0 + i / kgs of `src` (`kgroups`
// columns, `rblocks` row blocks); atoms outside them read as zeros.  Thread
// t of NT copies 16-byte chunks t, t + NT, ...
template <int NT>
__device__ __forceinline__ void load_atoms_plain(uint8_t *dst, const uint8_t *src, int count,
                                                 int kgs, int64_t rb0, int64_t kg0,
                                                 int64_t rblocks, int64_t kgroups, int tid) {
    const int chunks = count * 32;  // 512 / 16 per atom
    for (int c = tid; c < chunks; c += NT) {
        const int i = c >> 5, w = c & 31;
        const int64_t rb = rb0 + i / kgs, kg = kg0 + i % kgs;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (rb < rblocks && kg < kgroups)
            v = *reinterpret_cast<const uint4 *>(src + ((rb * kgroups + kg) * 512 + w * 16));
        *reinterpret_cast<uint4 *>(dst + c * 16) = v;
    }
}

template <Kind KD, int BN, bool PLAIN>
__global__ void __launch_bounds__(MxConfig<KD, BN>::threads(PLAIN), 1)
    tg_gemm_mx_kernel(const __grid_constant__ CUtensorMap tmap_a,
                      const __grid_constant__ CUtensorMap tmap_b,
                      const __grid_constant__ CUtensorMap tmap_sfa,
                      const __grid_constant__ CUtensorMap tmap_sfb, const GemmParams p) {
    using C = MxConfig<KD, BN>;
    constexpr int S = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: leader, 1: peer
    const uint32_t half = rank & 1u;
    const bool leader = half == 0;
    const int64_t pair = blockIdx.x / 2;
    const int64_t num_pairs = gridDim.x / 2;

    auto bar = [&](int i) -> uint32_t { return sbase + C::BAR_OFF + 8 * i; };
    auto a_stage = [&](int s) -> uint32_t { return sbase + C::A_OFF + s * C::A_BYTES; };
    auto b_stage = [&](int s) -> uint32_t { return sbase + C::B_OFF + s * C::B_BYTES; };
    auto sfa_stage = [&](int s) -> uint32_t { return sbase + C::SFA_OFF + s * C::SFA_BYTES; };
    auto sfb_stage = [&](int s) -> uint32_t { return sbase + C::SFB_OFF + s * C::SFB_BYTES; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
    const PairWaitCtl ctl{abort_flag, map_shared_rank(smem_u32(smem + C::MISC_OFF + 4), rank ^ 1u),
                          p.status, p.wait_limit_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            // Plain loads: every loader thread of both CTAs arrives.
            mbar_init(bar(C::FULL0 + s), PLAIN ? 2 * C::LOAD_WARPS * 32 : 1);
            mbar_init(bar(C::EMPTY0 + s), 1);
        }
        mbar_init(bar(C::ACCF), 1);
        mbar_init(bar(C::ACCE), 2 * C::EPI_WARPS);
        mbar_init(bar(C::DRAIN), 1);
        *abort_flag = 0;
        fence_mbar_init();
        if (!PLAIN) {
            prefetch_tensormap(&tmap_a);
            prefetch_tensormap(&tmap_b);
            prefetch_tensormap(&tmap_sfa);
            prefetch_tensormap(&tmap_sfb);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    // Programmatic dependent launch: each role waits for the preceding grid
    // before its first global-memory access (the producer after working out
    // its first tile).
    griddep_launch();
    const uint32_t tmem_base = *tmem_slot;
    const int nkb = p.num_k_blocks;

    if (PLAIN && warp >= C::NUM_WARPS) {
        // ------------------------------------------------------ plain-load producer (both CTAs)
        griddep_wait();
        constexpr int NT = C::LOAD_WARPS * 32;
        const int ltid = threadIdx.x - C::NUM_WARPS * 32;
        // Operand rows and K in bytes (packed FP4: two elements per byte).
        const int64_t lda_b = C::FP4 ? p.lda / 2 : p.lda, ldb_b = C::FP4 ? p.ldb / 2 : p.ldb;
        const int64_t sa_b = C::FP4 ? p.stride_a / 2 : p.stride_a;
        const int64_t sb_b = C::FP4 ? p.stride_b / 2 : p.stride_b;
        const int32_t k_bytes = C::FP4 ? p.k / 2 : p.k;
        const int64_t kgroups = ((int64_t)p.k + C::ATOM_K - 1) / C::ATOM_K;  // atom columns
        const int64_t rblocks_a = ((int64_t)p.m + BLOCK_M - 1) / BLOCK_M;
        const int64_t rblocks_b = ((int64_t)p.n + BLOCK_M - 1) / BLOCK_M;
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int64_t t = pair; ok && t < p.num_tiles; t += num_pairs) {
            int bt, mb, nb;
            batch_tile_coords(t, p, bt, mb, nb);
            const uint8_t *a_src = static_cast<const uint8_t *>(p.a_ptr) + (int64_t)bt * sa_b;
            const uint8_t *b_src = static_cast<const uint8_t *>(p.b_ptr) + (int64_t)bt * sb_b;
            const uint8_t *sfa_src =
                static_cast<const uint8_t *>(p.sfa_ptr) + (int64_t)bt * p.sfa_stride;
            const uint8_t *sfb_src =
                static_cast<const uint8_t *>(p.sfb_ptr) + (int64_t)bt * p.sfb_stride;
            const int32_t arow = mb * C::PAIR_M + (int32_t)half * BLOCK_M;
            const int32_t brow = nb * BN + (int32_t)half * C::B_ROWS;
            for (int kb = 0; kb < nkb; ++kb) {
                if (!pair_wait(bar(C::EMPTY0 + s), ph ^ 1, ctl, SITE_EMPTY)) { ok = false; break; }
                load_stage_plain<1, BLOCK_M, NT>(smem + C::A_OFF + s * C::A_BYTES, a_src, lda_b,
                                                 arow, p.m, kb * C::BK_UNITS, k_bytes, ltid);
                load_stage_plain<1, C::B_ROWS, NT>(smem + C::B_OFF + s * C::B_BYTES, b_src, ldb_b,
                                                   brow, p.n, kb * C::BK_UNITS, k_bytes, ltid);
                load_atoms_plain<NT>(smem + C::SFA_OFF + s * C::SFA_BYTES, sfa_src, C::KGS, C::KGS,
                                     mb * 2 + (int64_t)half, (int64_t)kb * C::KGS, rblocks_a,
                                     kgroups, ltid);
                if constexpr (C::REP) {
                    for (int a = 0; a < C::SFB_ATOMS; ++a)
                        for (int c = 0; c < 4; ++c)
                            load_atoms_plain<NT>(smem + C::SFB_OFF + s * C::SFB_BYTES +
                                                     a * C::REP_BYTES + c * C::ATOM_BYTES,
                                                 sfb_src, 1, 1, (int64_t)nb * C::SFB_ATOMS + a,
                                                 (int64_t)kb, rblocks_b, kgroups, ltid);
                } else {
                    load_atoms_plain<NT>(smem + C::SFB_OFF + s * C::SFB_BYTES, sfb_src,
                                         C::KGS * C::SFB_ATOMS, C::KGS,
                                         (int64_t)nb * C::SFB_ATOMS, (int64_t)kb * C::KGS,
                                         rblocks_b, kgroups, ltid);
                }
                fence_proxy_async_smem();
                if (leader) mbar_arrive(bar(C::FULL0 + s));
                else mbar_arrive_cluster(map_shared_rank(bar(C::FULL0 + s), 0));
                if (++s == S) { s = 0; ph ^= 1; }
            }
        }
    } else if (warp == 0) {
        // ------------------------------------------------------ TMA producer (both CTAs)
        if (!PLAIN && lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            bool waited = false;
            for (int64_t t = pair; ok && t < p.num_tiles; t += num_pairs) {
                int bt, mb, nb;
                batch_tile_coords(t, p, bt, mb, nb);
                if (!waited) {
                    griddep_wait();
                    waited = true;
                }
                const int32_t arow = mb * C::PAIR_M + (int32_t)half * BLOCK_M;
                const int32_t brow = nb * BN + (int32_t)half * C::B_ROWS;
                const int32_t ab = bt * p.a_bmul, bb = bt * p.b_bmul;
                // Scale atoms: this CTA's 128 A rows; all BN B rows.  An atom
                // column past the last one (FP4 with an odd count) reads as zeros.
                const int32_t sfa_rb = mb * 2 + (int32_t)half;
                const int32_t sfb_rb = nb * C::SFB_ATOMS;
                const int32_t sfa_b = bt * p.sfa_bmul, sfb_b = bt * p.sfb_bmul;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!pair_wait(bar(C::EMPTY0 + s), ph ^ 1, ctl, SITE_EMPTY)) { ok = false; break; }
                    const uint32_t full_leader = map_shared_rank(bar(C::FULL0 + s), 0);
                    if (leader) mbar_arrive_expect_tx(bar(C::FULL0 + s), 2 * C::STAGE_BYTES);
                    tma_load_3d_pair(a_stage(s), &tmap_a, full_leader, kb * C::BK_UNITS, arow, ab);
                    tma_load_3d_pair(b_stage(s), &tmap_b, full_leader, kb * C::BK_UNITS, brow, bb);
                    // One box per operand: the stage's KGS atom columns of the
                    // CTA's A row block, and of the tile's SFB_ATOMS B row blocks
                    // (REP: each B atom four times, one atom per box).
                    tma_load_4d_pair(sfa_stage(s), &tmap_sfa, full_leader, 0, kb * C::KGS, sfa_rb,
                                     sfa_b);
                    if constexpr (C::REP) {
                        // The map repeats each atom four times (a dimension of
                        // stride 0): both B atoms, four copies each, in one box.
                        tma_load_5d_pair(sfb_stage(s), &tmap_sfb, full_leader, 0, 0, kb, sfb_rb,
                                         sfb_b);
                    } else {
                        tma_load_4d_pair(sfb_stage(s), &tmap_sfb, full_leader, 0, kb * C::KGS,
                                         sfb_rb, sfb_b);
                    }
                    ++issued;
                    if (++s == S) { s = 0; ph ^= 1; }
                }
            }
            if (!ok && issued) pair_pause_ns(200000);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer (leader)
        griddep_wait();
        if (leader && lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t tl = 0;
            bool ok = true;
            for (int64_t t = pair; ok && t < p.num_tiles; t += num_pairs, ++tl) {
                if (!pair_wait(bar(C::ACCE), (tl & 1) ^ 1, ctl, SITE_ACC_EMPTY)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kb = 0; kb < nkb; ++kb) {
                    // Plain loads: the peer's loader threads completed the
                    // phase by release arrivals at cluster scope.
                    const bool got = PLAIN ? pair_wait_cluster(bar(C::FULL0 + s), ph, ctl, SITE_FULL)
                                           : pair_wait(bar(C::FULL0 + s), ph, ctl, SITE_FULL);
                    if (!got) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t slot = tmem_base + C::SF_COL0 + s * C::SLOT_COLS;
                    if constexpr (C::REP) {
                        // Both B atoms in one copy: lane L takes 32 bytes, row
                        // L % 32 of atom 0 (columns +0..3) and of atom 1 (+4..7),
                        // from the atoms' four-quarter copies 2 KB apart.
                        tmem_cp_32x128b_x4_pair(slot, smem_desc_rows16(sfa_stage(s)));
                        tmem_cp_128x256b_pair(slot + C::SFB_COL,
                                              smem_desc_k2(sfb_stage(s), C::REP_BYTES));
                    } else {
#pragma unroll
                        for (int g = 0; g < C::KGS; ++g) {
                            tmem_cp_32x128b_x4_pair(
                                slot + 4 * g, smem_desc_rows16(sfa_stage(s) + g * C::ATOM_BYTES));
#pragma unroll
                            for (int a = 0; a < C::SFB_ATOMS; ++a)
                                tmem_cp_32x128b_x4_pair(
                                    slot + C::SFB_COL + 4 * (g * C::SFB_ATOMS + a),
                                    smem_desc_rows16(sfb_stage(s) +
                                                     (a * C::KGS + g) * C::ATOM_BYTES));
                        }
                    }
                    const uint32_t a0 = a_stage(s), b0 = b_stage(s);
#pragma unroll
                    for (int kk = 0; kk < C::MMAS_PER_STAGE; ++kk) {
                        // Atom column of this MMA's scale blocks within the stage.
                        const int g = C::atom_col(kk);
                        const uint32_t sfa = slot + 4 * g;
                        const uint32_t sfb = slot + C::SFB_COL + 4 * C::SFB_ATOMS * g;
                        const uint64_t ad = smem_desc_sw128(a0 + kk * 32);
                        const uint64_t bd = smem_desc_sw128(b0 + kk * 32);
                        const uint32_t id = mx_idesc(C::IDESC, C::scale_id(kk));
                        if constexpr (C::NV) mma_nvf4_pair(tmem_base, ad, bd, id, sfa, sfb, (kb | kk) != 0);
                        else if constexpr (C::FP4) mma_mxf4_pair(tmem_base, ad, bd, id, sfa, sfb, (kb | kk) != 0);
                        else mma_mx_pair(tmem_base, ad, bd, id, sfa, sfb, (kb | kk) != 0);
                    }
                    mma_commit_pair_mcast(bar(C::EMPTY0 + s), 0x3);
                    if (++s == S) { s = 0; ph ^= 1; }
                }
                if (!ok) break;
                mma_commit_pair_mcast(bar(C::ACCF), 0x3);
            }
            if (!ok) {
                mma_commit_pair_mcast(bar(C::DRAIN), (uint16_t)(1u << rank));
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(bar(C::DRAIN), 0)) {
                    if (globaltimer_ns() - t0 > p.wait_limit_ns) {
                        atomicCAS(p.status, 0u, (uint32_t)SITE_DRAIN);
                        break;
                    }
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ epilogue (both CTAs)
        griddep_wait();
        const int q = warp & 3;
        const int row_in_half = q * 32 + lane;
        const int cbase = ((warp - 2) / 4) * C::COLS;
        uint32_t tl = 0;
        for (int64_t t = pair; t < p.num_tiles; t += num_pairs, ++tl) {
            int bt, mb, nb;
            batch_tile_coords(t, p, bt, mb, nb);
            if (!pair_wait(bar(C::ACCF), tl & 1, ctl, SITE_ACC_FULL)) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + cbase;
            uint32_t v[C::COLS / 32][32];
#pragma unroll
            for (int c = 0; c < C::COLS / 32; ++c) tmem_ld_32x32b_x32(taddr + c * 32, v[c]);
            tmem_ld_wait();
            // The accumulator is in registers: hand it back to the MMA.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader) mbar_arrive(bar(C::ACCE));
                else mbar_arrive_cluster_relaxed(map_shared_rank(bar(C::ACCE), 0));
            }
            const int32_t r = mb * C::PAIR_M + (int32_t)half * BLOCK_M + row_in_half;
            if (r < p.m) {
#pragma unroll
                for (int c = 0; c < C::COLS / 32; ++c)
                    epilogue_store(p, bt, r, nb * BN + cbase + c * 32, v[c]);
            }
        }
    }

    tc_fence_before();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace tg
