// CTA-pair variant of the persistent tcgen05 GEMM: one 256 x BN output tile
// per pair of CTAs on neighbouring SMs (a cluster of 2), with the MMA issued
// by the pair's leader as tcgen05.mma.cta_group::2.
//
// Each CTA stages its own 128 rows of the A-role tile and its own BN/2 rows of
// the B-role tile per K step (32 KB for BN = 256), so an SM moves half the B
// bytes of the single-CTA 128 x 256 tile through shared memory for the same
// FLOPs.  The accumulator rows 0-127 live in the leader's tensor memory, rows
// 128-255 in the peer's; each CTA's epilogue drains its own half.
//
// Synchronisation across the pair (all waits bounded, as in the single-CTA
// kernel):
//   full[s]   lives in the leader; the leader's producer arrives once with
//             the byte count of all four TMA loads of the stage (both CTAs'),
//             and every load signals its completion there (count 1 +
//             transaction bytes).  The peer's loads may land before the
//             leader's arrival; the phase cannot complete until it comes.
//   empty[s]  lives in both CTAs; the leader's commit after the stage's MMAs
//             arrives on both (multicast), so each producer refills its own
//             half of the stage.
//   acc_full  lives in both CTAs; the leader's commit at the end of a tile
//             arrives on both epilogues.
//   acc_empty lives in the leader; one lane of each epilogue warp of both
//             CTAs arrives (count 8) once its warp's rows have been read.
// The producers make no remote arrivals: a cluster-scope release per K step
// costs a memory barrier on the issuing thread and throttles the TMA issue.
// No TMA multicast is used: each CTA loads only its own rows.
#pragma once

#include <cstdint>
#include "tg_kernel.cuh"

namespace tg {

template <int BN>
struct PairStageCount {
    static constexpr int stage_bytes = (BLOCK_M + BN / 2) * ROW_BYTES;
    static constexpr int fit = (SMEM_LIMIT - 2048) / stage_bytes;
    static constexpr int value = fit > 8 ? 8 : fit;
};

template <Kind KD, int BN>
struct PairConfig {
    using T = KindTraits<KD>;
    static constexpr int BK = T::block_k;
    static constexpr int PAIR_M = 2 * BLOCK_M;      // 256 rows per pair tile
    static constexpr int B_ROWS = BN / 2;           // B-role rows staged by each CTA
    static constexpr int STAGES = PairStageCount<BN>::value;
    static constexpr int A_BYTES = BLOCK_M * ROW_BYTES;
    static constexpr int B_BYTES = B_ROWS * ROW_BYTES;
    static constexpr int A_OFF = 0;
    static constexpr int B_OFF = STAGES * A_BYTES;
    static constexpr int BAR_OFF = B_OFF + STAGES * B_BYTES;
    static constexpr int FULL0 = 0, EMPTY0 = STAGES;
    static constexpr int ACCF0 = 2 * STAGES, ACCE0 = 2 * STAGES + 2, DRAIN = 2 * STAGES + 4;
    static constexpr int NUM_BARS = 2 * STAGES + 5;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int NUM_WARPS = 6;
    static constexpr int NUM_THREADS = NUM_WARPS * 32;
    static constexpr int MMAS_PER_STAGE = BK / T::umma_k;
    // Instruction descriptor as in the single-CTA kernel with M = 256.
    static constexpr uint32_t IDESC = (1u << 4) | (T::fmt << 7) | (T::fmt << 10) |
                                      ((uint32_t)(BN >> 3) << 17) |
                                      ((uint32_t)(PAIR_M >> 4) << 24);
    static_assert(KD != Kind::TF32, "the pair kernel covers the 16-bit kinds");
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory budget");
    static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "UMMA N for M = 256");
    static_assert(TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM allocation");
};

struct PairWaitCtl {
    volatile int *abort_flag;
    uint32_t peer_abort;  // shared::cluster address of the peer CTA's abort flag
    uint32_t *status;
    uint64_t limit_ns;
};

__device__ __forceinline__ void pair_raise_abort(const PairWaitCtl &c, uint32_t site) {
    *c.abort_flag = 1;
    st_cluster_u32(c.peer_abort, 1u);
    atomicCAS(c.status, 0u, site);
}

__device__ __forceinline__ bool pair_wait(uint32_t bar, uint32_t parity, const PairWaitCtl &c,
                                          uint32_t site) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*c.abort_flag) return false;
        if (globaltimer_ns() - t0 > c.limit_ns) {
            pair_raise_abort(c, site);
            return false;
        }
    }
}

__device__ __forceinline__ void pair_pause_ns(uint64_t ns) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < ns) {
    }
}

template <Kind KD, int BN>
__global__ void __launch_bounds__(PairConfig<KD, BN>::NUM_THREADS, 1)
    tg_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_b, const GemmParams p) {
    using C = PairConfig<KD, BN>;
    constexpr int S = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int64_t pair = blockIdx.x >> 1;
    const int64_t num_pairs = gridDim.x >> 1;

    auto bar = [&](int i) -> uint32_t { return sbase + C::BAR_OFF + 8 * i; };
    auto a_stage = [&](int s) -> uint32_t { return sbase + C::A_OFF + s * C::A_BYTES; };
    auto b_stage = [&](int s) -> uint32_t { return sbase + C::B_OFF + s * C::B_BYTES; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
    const PairWaitCtl ctl{abort_flag, map_shared_rank(smem_u32(smem + C::MISC_OFF + 4), rank ^ 1u),
                          p.status, p.wait_limit_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar(C::FULL0 + s), 1);
            mbar_init(bar(C::EMPTY0 + s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar(C::ACCF0 + a), 1);
            mbar_init(bar(C::ACCE0 + a), 2 * 4);
        }
        mbar_init(bar(C::DRAIN), 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_b);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();  // both CTAs' barriers initialised, tensor memory allocated
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int nkb = p.num_k_blocks;

    if (warp == 0) {
        // ------------------------------------------------------ producer (both CTAs)
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int64_t t = pair; ok && t < p.num_tiles; t += num_pairs) {
                int mb, nb;
                tile_coords(t, p, mb, nb);
                const int32_t arow = mb * C::PAIR_M + (int32_t)rank * BLOCK_M;
                const int32_t brow = nb * BN + (int32_t)rank * C::B_ROWS;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!pair_wait(bar(C::EMPTY0 + s), ph ^ 1, ctl, SITE_EMPTY)) { ok = false; break; }
                    const uint32_t full_leader = map_shared_rank(bar(C::FULL0 + s), 0);
                    if (leader) mbar_arrive_expect_tx(bar(C::FULL0 + s), 2 * (C::A_BYTES + C::B_BYTES));
                    tma_load_2d_pair(a_stage(s), &tmap_a, full_leader, kb * C::BK, arow);
                    tma_load_2d_pair(b_stage(s), &tmap_b, full_leader, kb * C::BK, brow);
                    ++issued;
                    if (++s == S) { s = 0; ph ^= 1; }
                }
            }
            if (!ok && issued) {
                // Copies already issued land within microseconds; let them
                // finish before this CTA can leave (their barriers may be the
                // peer's, which this thread cannot poll).
                pair_pause_ns(200000);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer (leader)
        if (leader && lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t tl = 0;
            bool ok = true;
            for (int64_t t = pair; ok && t < p.num_tiles; t += num_pairs, ++tl) {
                const uint32_t acc = tl & 1, use = tl >> 1;
                if (!pair_wait(bar(C::ACCE0 + acc), (use & 1) ^ 1, ctl, SITE_ACC_EMPTY)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!pair_wait(bar(C::FULL0 + s), ph, ctl, SITE_FULL)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a0 = a_stage(s), b0 = b_stage(s);
#pragma unroll
                    for (int kk = 0; kk < C::MMAS_PER_STAGE; ++kk) {
                        mma_f16_pair(d_tmem, smem_desc_sw128(a0 + kk * 32),
                                     smem_desc_sw128(b0 + kk * 32), C::IDESC, (kb | kk) != 0);
                    }
                    mma_commit_pair_mcast(bar(C::EMPTY0 + s), (uint16_t)0x3);
                    if (++s == S) { s = 0; ph ^= 1; }
                }
                if (!ok) break;
                mma_commit_pair_mcast(bar(C::ACCF0 + acc), (uint16_t)0x3);
            }
            if (!ok) {
                mma_commit_pair_mcast(bar(C::DRAIN), (uint16_t)0x1);
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
        const int q = warp & 3;
        const int row_in_half = q * 32 + lane;
        uint32_t tl = 0;
        for (int64_t t = pair; t < p.num_tiles; t += num_pairs, ++tl) {
            int mb, nb;
            tile_coords(t, p, mb, nb);
            const uint32_t acc = tl & 1, use = tl >> 1;
            if (!pair_wait(bar(C::ACCF0 + acc), use & 1, ctl, SITE_ACC_FULL)) break;
            tc_fence_after();
            const int32_t r = mb * C::PAIR_M + (int32_t)rank * BLOCK_M + row_in_half;
            const bool row_ok = r < p.m;
            float *drow = p.d + (int64_t)r * p.d_row_stride;
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(taddr + c0, v);
                tmem_ld_wait();
                const int32_t col0 = nb * BN + c0;
                if (row_ok) {
                    if (p.vector_store && col0 + 32 <= p.n) {
                        float4 *dst = reinterpret_cast<float4 *>(drow + col0);
#pragma unroll
                        for (int j = 0; j < 32; j += 4) {
                            dst[j / 4] = make_float4(
                                apply_epilogue(__uint_as_float(v[j]), p.alpha, p.relu),
                                apply_epilogue(__uint_as_float(v[j + 1]), p.alpha, p.relu),
                                apply_epilogue(__uint_as_float(v[j + 2]), p.alpha, p.relu),
                                apply_epilogue(__uint_as_float(v[j + 3]), p.alpha, p.relu));
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            if (col0 + j < p.n) {
                                drow[(int64_t)(col0 + j) * p.d_col_stride] =
                                    apply_epilogue(__uint_as_float(v[j]), p.alpha, p.relu);
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(map_shared_rank(bar(C::ACCE0 + acc), 0));
        }
    }

    tc_fence_before();
    cluster_sync_all();  // neither CTA leaves while the pair may still touch its memory
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace tg
