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
//             CTAs arrives (count 16) once its warp's part has been read.
// The producers make no remote arrivals: a cluster-scope release per K step
// costs a memory barrier on the issuing thread and throttles the TMA issue.
// With one pair per cluster (MC = 1) each CTA loads only its own rows; with
// two (MC = 2, below) the pairs share their A rows by TMA multicast.  Work
// is a static persistent sequence of units; or (MC = 1, p.dynamic) one
// cluster per tile with tiles taken over through cluster launch control; or
// (MC = 1, p.ticket) a persistent grid whose pairs take their first unit
// statically and claim every later one, in order, from a counter in global
// memory, so that pairs that run ahead take more of the work.  The claimed
// unit reaches every role of both CTAs through the same ring of answer slots
// that cluster launch control fills.
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
    // Dynamic schedule: a ring of CLC_SLOTS launch-control answers, each with
    // a full barrier (answer landed, in both CTAs) and an empty barrier (in
    // the leader: every reader of both CTAs is done with it).
    static constexpr int CLC_SLOTS = 4;
    static constexpr int CLCF0 = 2 * STAGES + 5, CLCE0 = CLCF0 + CLC_SLOTS;
    static constexpr int NUM_BARS = CLCE0 + CLC_SLOTS;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int CLC_OFF = (MISC_OFF + 16 + 15) / 16 * 16;
    // Ticket schedule: the leader writes each claimed unit here, then copies
    // it into the answer slot of both CTAs.
    static constexpr int TICKET_OFF = CLC_OFF + 16 * CLC_SLOTS;
    static constexpr int SMEM_BYTES = TICKET_OFF + 16 * CLC_SLOTS + 1024;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int EPI_WARPS = 8;  // two per tensor-memory lane quarter
    static constexpr int NUM_WARPS = 2 + EPI_WARPS;
    static constexpr int NUM_THREADS = NUM_WARPS * 32;
    static constexpr int MMAS_PER_STAGE = BK / T::umma_k;
    // Readers of each answer: producer, MMA thread and epilogue warps of the
    // leader; producer and epilogue warps of the peer.
    static constexpr int CLC_READERS = 2 * (1 + EPI_WARPS) + 1;
    // Instruction descriptor as in the single-CTA kernel with M = 256.
    static constexpr uint32_t IDESC = (1u << 4) | (T::fmt << 7) | (T::fmt << 10) |
                                      ((uint32_t)(BN >> 3) << 17) |
                                      ((uint32_t)(PAIR_M >> 4) << 24);
    static_assert(KD != Kind::TF32, "the pair kernel covers the 16-bit and 8-bit kinds");
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

// pair_wait for a phase completed by release arrivals of the other CTA's
// threads (acquire at cluster scope).
__device__ __forceinline__ bool pair_wait_cluster(uint32_t bar, uint32_t parity,
                                                  const PairWaitCtl &c, uint32_t site) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
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

// Work units.  With P pairs and T tiles, the first T - R tiles (R = T mod P)
// are whole units; when the split is on, each of the last R tiles is cut
// into S contiguous K segments (S = min(P / R, split_max, K blocks / 8), so the
// R * S tail units fit in one round of the P pairs).  Pair p takes units
// p, p + P, ...; a tail tile's segments land on consecutive pairs of the
// last round.  Segments 0 .. S-2 store their FP32 partial accumulators to
// the workspace and raise a flag; segment S-1 (on the highest-numbered of
// those pairs, so it only waits on pairs dispatched before it) adds the
// partials in segment order, applies the epilogue and stores D, so the
// summation order is fixed and the result is deterministic.  With S = 2 the
// two segments instead exchange halves: each writes the partial sums of the
// columns the other finishes, raises its flag, waits for the other's flag,
// adds the other's partials to its own half and stores it.  Each side then
// moves half the bytes of a one-sided finish, and both sides' stores run at
// once.  Both segments write before they wait, and both are dispatched in
// the same round (static) or as consecutive claims (ticket), so neither
// waits on work that has not been handed out.
// A K segment spans at least this many K blocks, so that a segment's MMA
// work outweighs the finisher's read of one partial tile.
constexpr int SPLIT_MIN_KBLOCKS = 8;

struct UnitPlan {
    int64_t tiles, whole, units;  // tiles, whole-tile units, total units
    int32_t segs;                 // K segments per tail tile (1: no split)
};

__device__ __forceinline__ UnitPlan make_unit_plan(const GemmParams &p, int64_t pairs) {
    UnitPlan u;
    u.tiles = p.num_tiles;
    u.segs = 1;
    const int64_t rem = p.num_tiles % pairs;
    if (p.split_max > 1 && rem > 0) {
        int64_t s = pairs / rem;
        if (s > p.split_max) s = p.split_max;
        if (s > p.num_k_blocks / SPLIT_MIN_KBLOCKS) s = p.num_k_blocks / SPLIT_MIN_KBLOCKS;
        if (s > 1 && rem * (s - 1) <= p.ws_tiles) u.segs = (int32_t)s;
    }
    u.whole = u.segs > 1 ? p.num_tiles - rem : p.num_tiles;
    u.units = u.whole + (p.num_tiles - u.whole) * u.segs;
    return u;
}

struct Unit {
    int64_t tile;
    int32_t k0, k1;  // K blocks [k0, k1)
    int32_t seg;     // -1: whole tile; else segment index of a tail tile
    int64_t tail;    // tail-tile index (seg >= 0)
};

__device__ __forceinline__ Unit decode_unit(const UnitPlan &up, int64_t u, int nkb) {
    Unit r;
    if (u < up.whole) {
        r.tile = u; r.k0 = 0; r.k1 = nkb; r.seg = -1; r.tail = 0;
    } else {
        const int64_t j = u - up.whole;
        r.tail = j / up.segs;
        r.seg = (int32_t)(j % up.segs);
        r.tile = up.whole + r.tail;
        r.k0 = (int32_t)((int64_t)r.seg * nkb / up.segs);
        r.k1 = (int32_t)((int64_t)(r.seg + 1) * nkb / up.segs);
    }
    return r;
}

// MC = 1: a cluster is one CTA pair.  MC = 2: a cluster of four CTAs is two
// pairs working on the same 256 A-role rows and neighbouring N blocks (pair
// q of the cluster takes N block MC * nbc + q).  Then each CTA loads half of
// its 128 A rows and multicasts them to itself and to the CTA holding the
// same rows in the other pair, so each CTA moves 24 KB instead of 32 KB per
// K step through L2; a stage is refilled only after both pairs' MMAs are
// done with it (its empty barrier takes one arrival from each pair leader).
template <Kind KD, int BN, int MC>
__global__ void __launch_bounds__(PairConfig<KD, BN>::NUM_THREADS, 1)
    tg_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_b, const GemmParams p) {
    using C = PairConfig<KD, BN>;
    constexpr int S = C::STAGES;
    static_assert(MC == 1 || MC == 2, "one or two pairs per cluster");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();     // 0 .. 2*MC-1
    const uint32_t half = rank & 1u;              // 0: pair leader, 1: pair peer
    const uint32_t pic = rank >> 1;               // pair within the cluster
    const uint32_t lead_rank = rank & ~1u;
    const bool leader = half == 0;
    const int64_t pair = blockIdx.x / (2 * MC);   // cluster index (work-unit stride)
    const int64_t num_pairs = gridDim.x / (2 * MC);
    constexpr uint16_t ALL_CTAS = (uint16_t)((1u << (2 * MC)) - 1u);
    const uint16_t pair_ctas = (uint16_t)(0x3u << (2 * pic));

    auto bar = [&](int i) -> uint32_t { return sbase + C::BAR_OFF + 8 * i; };
    auto a_stage = [&](int s) -> uint32_t { return sbase + C::A_OFF + s * C::A_BYTES; };
    auto b_stage = [&](int s) -> uint32_t { return sbase + C::B_OFF + s * C::B_BYTES; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
    volatile int *fin_ready = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 8);
    const PairWaitCtl ctl{abort_flag, map_shared_rank(smem_u32(smem + C::MISC_OFF + 4), rank ^ 1u),
                          p.status, p.wait_limit_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar(C::FULL0 + s), 1);
            mbar_init(bar(C::EMPTY0 + s), MC);  // one arrival per pair leader
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar(C::ACCF0 + a), 1);
            mbar_init(bar(C::ACCE0 + a), 2 * C::EPI_WARPS);
        }
        mbar_init(bar(C::DRAIN), 1);
        for (int c = 0; c < C::CLC_SLOTS; ++c) {
            mbar_init(bar(C::CLCF0 + c), 1);
            mbar_init(bar(C::CLCE0 + c), C::CLC_READERS);
        }
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
    // Programmatic dependent launch: every role waits for the preceding grid
    // before its first global-memory access (the producer after working out
    // its first unit, so that its first load leaves right after the wait).
    griddep_launch();
    const uint32_t tmem_base = *tmem_slot;
    const int nkb = p.num_k_blocks;
    const UnitPlan up = make_unit_plan(p, num_pairs);
    // Work sequence.  Static: units pair, pair + P, ...  Dynamic (MC == 1,
    // no split): this cluster's own tile, then the tile of each cluster that
    // launch control cancelled for it, until an answer says none was left.
    const bool dyn = MC == 1 && p.dynamic != 0;
    // Ticket schedule: every pair has a first unit (units >= pairs), so each
    // makes exactly one failing claim and the claims of a launch number
    // exactly `units`; the last one (value units - 1) resets the counter.
    const bool tick = MC == 1 && !dyn && p.ticket != nullptr && up.units >= num_pairs;
    const bool ring = dyn || tick;
    const int64_t first_unit = dyn ? (int64_t)(blockIdx.x / 2) : pair;
    // Read answer `step` (waiting for it), release its slot, return the next
    // unit (-1: no more work; -2: the wait gave up).  One thread per reader.
    auto clc_read = [&](int64_t step) -> int64_t {
        const int slot = (int)(step % C::CLC_SLOTS);
        int64_t next = -2;
        if (pair_wait(bar(C::CLCF0 + slot), (uint32_t)((step / C::CLC_SLOTS) & 1), ctl,
                      SITE_SCHED)) {
            const volatile uint64_t *r =
                reinterpret_cast<const volatile uint64_t *>(smem + C::CLC_OFF + 16 * slot);
            if (tick) {
                next = (int64_t)r[0];  // the claimed unit, or -1
            } else {
                const int32_t x = clc_cancelled_x(r[0], r[1]);
                next = x >= 0 ? (int64_t)(x / 2) : -1;
            }
        }
        if (leader) mbar_arrive(bar(C::CLCE0 + slot));
        else mbar_arrive_cluster(map_shared_rank(bar(C::CLCE0 + slot), lead_rank));
        return next;
    };
    // The same for a whole warp: lane 0 reads, every lane gets the result.
    auto clc_read_warp = [&](int64_t step) -> int64_t {
        int64_t next = 0;
        if (lane == 0) next = clc_read(step);
        return __shfl_sync(0xffffffffu, next, 0);
    };

    if (warp == 0) {
        // ------------------------------------------------------ producer (both CTAs)
        if (lane == 0) {
            const uint64_t pol_a = l2_policy_evict_last();
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            int64_t step = 0;
            bool waited = false;
            for (int64_t u = first_unit; ok && u >= 0 && u < up.units;) {
                const Unit un = decode_unit(up, u, nkb);
                int bt, mb, nbc;
                batch_tile_coords(un.tile, p, bt, mb, nbc);
                if (!waited) {
                    griddep_wait();  // also orders the ticket claims after the previous launch
                    waited = true;
                }
                if (ring) {
                    // Ask for the unit after this one (answer `step`), into a
                    // slot all readers have released.
                    const int slot = (int)(step % C::CLC_SLOTS);
                    mbar_arrive_expect_tx(bar(C::CLCF0 + slot), 16);
                    if (leader) {
                        if (step >= C::CLC_SLOTS &&
                            !pair_wait(bar(C::CLCE0 + slot),
                                       (uint32_t)(((step / C::CLC_SLOTS) - 1) & 1), ctl, SITE_SCHED)) {
                            ok = false;
                            break;
                        }
                        if (dyn) {
                            clc_try_cancel_all(sbase + C::CLC_OFF + 16 * slot, bar(C::CLCF0 + slot));
                        } else {
                            // Claim the next unit in order; the answer lands in
                            // both CTAs' slot as 16 transaction bytes, like a
                            // launch-control answer.
                            const uint32_t v = atomicAdd(p.ticket, 1u);
                            int64_t next = num_pairs + (int64_t)v;
                            if (next >= up.units) {
                                next = -1;
                                if ((int64_t)v == up.units - 1) atomicExch(p.ticket, 0u);
                            }
                            volatile int64_t *stg =
                                reinterpret_cast<volatile int64_t *>(smem + C::TICKET_OFF + 16 * slot);
                            stg[0] = next;
                            stg[1] = 0;
                            fence_proxy_async_smem();
                            const uint32_t src = sbase + C::TICKET_OFF + 16 * slot;
                            const uint32_t dst = sbase + C::CLC_OFF + 16 * slot;
                            const uint32_t fb = bar(C::CLCF0 + slot);
                            bulk_copy_s2cluster(map_shared_rank(dst, rank), src, 16,
                                                map_shared_rank(fb, rank));
                            bulk_copy_s2cluster(map_shared_rank(dst, rank ^ 1u), src, 16,
                                                map_shared_rank(fb, rank ^ 1u));
                        }
                    }
                }
                const int nb = nbc * MC + (int)pic;
                const int32_t arow = mb * C::PAIR_M + (int32_t)half * BLOCK_M;
                const int32_t brow = nb * BN + (int32_t)half * C::B_ROWS;
                const int32_t ab = bt * p.a_bmul, bb = bt * p.b_bmul;
                const bool down = p.k_snake && ((un.tile / num_pairs) & 1);
                for (int i = 0; i < un.k1 - un.k0; ++i) {
                    const int kb = down ? un.k1 - 1 - i : un.k0 + i;
                    if (!pair_wait(bar(C::EMPTY0 + s), ph ^ 1, ctl, SITE_EMPTY)) { ok = false; break; }
                    const uint32_t full_leader = map_shared_rank(bar(C::FULL0 + s), lead_rank);
                    if (leader) mbar_arrive_expect_tx(bar(C::FULL0 + s), 2 * (C::A_BYTES + C::B_BYTES));
                    if constexpr (MC == 2) {
                        // Half of this CTA's A rows, to this CTA and its partner.
                        constexpr int HALF_ROWS = BLOCK_M / 2;
                        tma_load_3d_pair_mcast(a_stage(s) + pic * HALF_ROWS * ROW_BYTES, &tmap_a,
                                               full_leader, kb * C::BK,
                                               arow + (int32_t)pic * HALF_ROWS, ab,
                                               (uint16_t)((1u << rank) | (1u << (rank ^ 2u))));
                        tma_load_3d_pair(b_stage(s), &tmap_b, full_leader, kb * C::BK, brow, bb);
                    } else if (p.l2_hint) {
                        tma_load_3d_pair_hint(a_stage(s), &tmap_a, full_leader, kb * C::BK, arow,
                                              ab, pol_a);
                        tma_load_3d_pair(b_stage(s), &tmap_b, full_leader, kb * C::BK, brow, bb);
                    } else {
                        tma_load_3d_pair(a_stage(s), &tmap_a, full_leader, kb * C::BK, arow, ab);
                        tma_load_3d_pair(b_stage(s), &tmap_b, full_leader, kb * C::BK, brow, bb);
                    }
                    ++issued;
                    if (++s == S) { s = 0; ph ^= 1; }
                }
                if (!ok) break;
                u = ring ? clc_read(step++) : u + num_pairs;
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
        griddep_wait();
        if (leader && lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t tl = 0;
            bool ok = true;
            int64_t step = 0;
            for (int64_t u = first_unit; ok && u >= 0 && u < up.units; ++tl) {
                const Unit un = decode_unit(up, u, nkb);
                const uint32_t acc = tl & 1, use = tl >> 1;
                if (!pair_wait(bar(C::ACCE0 + acc), (use & 1) ^ 1, ctl, SITE_ACC_EMPTY)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                // K blocks in the producer's order (see k_snake); the first
                // one initialises the accumulator.
                for (int i = 0; i < un.k1 - un.k0; ++i) {
                    if (!pair_wait(bar(C::FULL0 + s), ph, ctl, SITE_FULL)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a0 = a_stage(s), b0 = b_stage(s);
#pragma unroll
                    for (int kk = 0; kk < C::MMAS_PER_STAGE; ++kk) {
                        mma_kind_pair<KD>(d_tmem, smem_desc_sw128(a0 + kk * 32),
                                     smem_desc_sw128(b0 + kk * 32), C::IDESC,
                                     (i != 0) || (kk != 0));
                    }
                    // Every CTA of the cluster may write this stage (multicast).
                    mma_commit_pair_mcast(bar(C::EMPTY0 + s), ALL_CTAS);
                    if (++s == S) { s = 0; ph ^= 1; }
                }
                if (!ok) break;
                mma_commit_pair_mcast(bar(C::ACCF0 + acc), pair_ctas);
                u = ring ? clc_read(step++) : u + num_pairs;
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
        constexpr int EPI_THREADS = C::EPI_WARPS * 32;
        const int etid = threadIdx.x - 64;  // 0 .. EPI_THREADS-1 over the epilogue warps
        constexpr int COLS = BN / (C::EPI_WARPS / 4);  // columns of this warp
        const int cbase = ((warp - 2) / 4) * COLS;
        uint32_t tl = 0;
        int64_t step = 0;
        for (int64_t u = first_unit; u >= 0 && u < up.units; ++tl) {
            const Unit un = decode_unit(up, u, nkb);
            int bt, mb, nbc;
            batch_tile_coords(un.tile, p, bt, mb, nbc);
            const int nb = nbc * MC + (int)pic;
            const uint32_t acc = tl & 1, use = tl >> 1;
            const bool got = pair_wait(bar(C::ACCF0 + acc), use & 1, ctl, SITE_ACC_FULL);
            // With split tiles the epilogue warps meet on named barriers, so
            // they leave together: if any thread's wait gave up, all stop.
            if (up.segs > 1 ? named_bar_any(2, EPI_THREADS, !got) : !got) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
            // Partial tile `k` of this tail tile, this CTA's half: column-major
            // 128 rows x BN columns of FP32.
            auto part = [&](int32_t k) -> float * {
                const int64_t pidx = un.tail * (up.segs - 1) + k;
                return p.ws + ((pidx * 2 + half) * BN) * (int64_t)BLOCK_M;
            };
            auto flag = [&](int32_t k) -> uint32_t * {
                return p.flags + (un.tail * (up.segs - 1) + k) * 2 + half;
            };
            if (un.seg >= 0 && up.segs == 2) {
                // Exchange (two segments): this segment finishes column half
                // `sg` of each warp's range and hands the other half over.
                constexpr int HALF = COLS / 2;
                const int32_t sg = un.seg, other = 1 - sg;
                const int grp = (warp - 2) / 4;  // this warp's column range
                // Partials of segment k: the half it hands over, column-major
                // 128 rows x BN/2 columns of FP32 (group-major columns).
                auto xpart = [&](int32_t k) -> float * {
                    return p.ws + ((un.tail * 2 + half) * BN + k * (BN / 2)) * (int64_t)BLOCK_M;
                };
                auto xflag = [&](int32_t k) -> uint32_t * {
                    return p.flags + (un.tail * 2 + half) * 2 + k;
                };
                float *mine = xpart(sg) + (int64_t)grp * HALF * BLOCK_M + row_in_half;
#pragma unroll 1
                for (int c0 = 0; c0 < HALF; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(taddr + cbase + other * HALF + c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        __stcg(mine + (int64_t)(c0 + j) * BLOCK_M, __uint_as_float(v[j]));
                }
                __threadfence();
                named_bar_sync(1, EPI_THREADS);
                if (etid == 0) st_release_gpu_u32(xflag(sg), 1u);
                bool ready = true;
                if (etid == 0) {
                    const uint64_t t0 = globaltimer_ns();
                    while (ld_acquire_gpu_u32(xflag(other)) == 0u) {
                        if (*abort_flag || globaltimer_ns() - t0 > p.wait_limit_ns) {
                            if (!*abort_flag) pair_raise_abort(ctl, SITE_PARTIAL);
                            ready = false;
                            break;
                        }
                    }
                    *fin_ready = ready ? 1 : 0;
                }
                named_bar_sync(1, EPI_THREADS);
                ready = *fin_ready != 0;
                if (ready) (void)ld_acquire_gpu_u32(xflag(other));
                const int32_t r = mb * C::PAIR_M + (int32_t)half * BLOCK_M + row_in_half;
                const bool row_ok = r < p.m;
                const float *theirs = xpart(other) + (int64_t)grp * HALF * BLOCK_M + row_in_half;
                // All of this thread's partials are requested at once: the
                // other segment's pair may sit on the other die, and one
                // round trip per 32 columns would put that latency in series.
                float pv[HALF];
                if (ready) {
#pragma unroll
                    for (int j = 0; j < HALF; ++j) pv[j] = __ldcg(theirs + (int64_t)j * BLOCK_M);
                }
#pragma unroll
                for (int c0 = 0; c0 < HALF; c0 += 32) {
                    if (!ready) break;
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(taddr + cbase + sg * HALF + c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        v[j] = __float_as_uint(__uint_as_float(v[j]) + pv[c0 + j]);
                    if (row_ok) epilogue_store(p, bt, r, nb * BN + cbase + sg * HALF + c0, v);
                }
                // The other segment's flag was raised for this launch only:
                // put it back to zero (this side is its only reader).
                if (etid == 0 && ready) *xflag(other) = 0u;
            } else if (un.seg >= 0 && un.seg < up.segs - 1) {
                // Writer: raw FP32 partial sums to the workspace, then the flag.
                float *dst = part(un.seg);
#pragma unroll 1
                for (int c0 = cbase; c0 < cbase + COLS; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(taddr + c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        __stcg(dst + (int64_t)(c0 + j) * BLOCK_M + row_in_half, __uint_as_float(v[j]));
                }
                __threadfence();
                named_bar_sync(1, EPI_THREADS);
                if (etid == 0) st_release_gpu_u32(flag(un.seg), 1u);
            } else {
                const bool finisher = un.seg >= 0;  // last segment of a tail tile
                bool ready = true;
                if (finisher) {
                    // Wait (bounded) for the earlier segments' partials.
                    if (etid == 0) {
                        const uint64_t t0 = globaltimer_ns();
                        for (int32_t k = 0; k < up.segs - 1 && ready; ++k) {
                            while (ld_acquire_gpu_u32(flag(k)) == 0u) {
                                if (*abort_flag || globaltimer_ns() - t0 > p.wait_limit_ns) {
                                    if (!*abort_flag) pair_raise_abort(ctl, SITE_PARTIAL);
                                    ready = false;
                                    break;
                                }
                            }
                        }
                    }
                    if (etid == 0) *fin_ready = ready ? 1 : 0;
                    named_bar_sync(1, EPI_THREADS);
                    ready = *fin_ready != 0;
                    if (ready) {
                        for (int32_t k = 0; k < up.segs - 1; ++k) (void)ld_acquire_gpu_u32(flag(k));
                    }
                }
                const int32_t r = mb * C::PAIR_M + (int32_t)half * BLOCK_M + row_in_half;
                const bool row_ok = r < p.m;
#pragma unroll 1
                for (int c0 = cbase; ready && c0 < cbase + COLS; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(taddr + c0, v);
                    tmem_ld_wait();
                    if (finisher) {
                        for (int32_t k = 0; k < up.segs - 1; ++k) {
                            const float *src = part(k) + (int64_t)c0 * BLOCK_M + row_in_half;
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                v[j] = __float_as_uint(__uint_as_float(v[j]) +
                                                       __ldcg(src + (int64_t)j * BLOCK_M));
                        }
                    }
                    if (row_ok) epilogue_store(p, bt, r, nb * BN + c0, v);
                }
                if (finisher) {
                    // Leave the flags at zero for the next launch.
                    named_bar_sync(1, EPI_THREADS);
                    if (etid == 0 && ready)
                        for (int32_t k = 0; k < up.segs - 1; ++k) *flag(k) = 0u;
                }
            }
            tc_fence_before();
            __syncwarp();
            // Release the accumulator to the leader's MMA.  The leader's warps
            // arrive locally; the peer's arrive remotely without a cluster-scope
            // release, which would first wait for this warp's D stores to drain.
            if (lane == 0) {
                if (leader) mbar_arrive(bar(C::ACCE0 + acc));
                else mbar_arrive_cluster_relaxed(map_shared_rank(bar(C::ACCE0 + acc), lead_rank));
            }
            u = ring ? clc_read_warp(step++) : u + num_pairs;
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
