// Kernel instantiation and launch for one operand kind; included once by each
// tg_inst_<kind>.cu so the operand kinds compile in parallel.
#pragma once

#include <atomic>
#include <cstdio>
#include <cstdlib>
#include "tg_launch.h"

namespace tg {

template <Kind KD, int BN, bool PLAIN>
static cudaError_t launch_one(const LaunchArgs &a) {
    using C = Config<KD, BN>;
    auto kernel = tg_gemm_kernel<KD, BN, PLAIN>;
    // The dynamic shared-memory opt-in is a per-device function attribute:
    // set it once per device.
    static std::atomic<uint64_t> configured{0};
    const uint64_t bit = (a.device >= 0 && a.device < 64) ? (1ull << a.device) : 0;
    if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(a.grid, 1, 1);
    cfg.blockDim = dim3(C::threads(PLAIN), 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e2 = cudaLaunchKernelEx(&cfg, kernel, a.map_a, a.map_b, a.p);
    if (e2 != cudaSuccess) return e2;
    return cudaGetLastError();
}

// CTA-pair kernel: cluster of 2 along x; the grid is clamped to the number
// of pairs the device can hold at once (queried once per device).
template <Kind KD, int BN, int MC>
static cudaError_t launch_pair(const LaunchArgs &a) {
    using C = PairConfig<KD, BN>;
    constexpr int CL = 2 * MC;  // CTAs per cluster
    auto kernel = tg_gemm_pair_kernel<KD, BN, MC>;
    static std::atomic<uint64_t> configured{0};
    static int max_clusters[64] = {0};
    const uint64_t bit = (a.device >= 0 && a.device < 64) ? (1ull << a.device) : 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(C::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        int n = 0;
        cfg.gridDim = dim3(CL, 1, 1);
        e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        if (bit) max_clusters[a.device] = n;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    int grid = a.grid - a.grid % CL;
    // A dynamic schedule launches one cluster per tile (not capped: clusters
    // that do not fit wait, and running clusters may take over their tiles).
    const int cap = bit && !a.p.dynamic ? CL * max_clusters[a.device] : grid;
    if (grid > cap) grid = cap;
    if (grid < CL) grid = CL;
    cfg.gridDim = dim3(grid, 1, 1);
    if (std::getenv("TG_LOG"))
        std::fprintf(stderr, "tg_gemm: pair kernel BN=%d MC=%d grid=%d (planned %d, %d co-resident clusters)\n",
                     BN, MC, grid, a.grid, bit ? max_clusters[a.device] : -1);
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, a.map_a, a.map_b, a.p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <Kind KD>
static cudaError_t launch_kind(const LaunchArgs &a) {
    if (a.pair) {
        if constexpr (KD == Kind::TF32) {
            return cudaErrorInvalidValue;
        } else {
            if (a.plain_loads) return cudaErrorInvalidValue;
            if (a.mc == 2) {
                if (a.block_n == 256) return launch_pair<KD, 256, 2>(a);
                if (a.block_n == 128) return launch_pair<KD, 128, 2>(a);
            } else {
                if (a.block_n == 256) return launch_pair<KD, 256, 1>(a);
                if (a.block_n == 128) return launch_pair<KD, 128, 1>(a);
            }
            return cudaErrorInvalidValue;
        }
    }
    switch (a.block_n) {
    case 64:
        return a.plain_loads ? launch_one<KD, 64, true>(a) : launch_one<KD, 64, false>(a);
    case 128:
        return a.plain_loads ? launch_one<KD, 128, true>(a) : launch_one<KD, 128, false>(a);
    case 256:
        return a.plain_loads ? launch_one<KD, 256, true>(a) : launch_one<KD, 256, false>(a);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace tg
