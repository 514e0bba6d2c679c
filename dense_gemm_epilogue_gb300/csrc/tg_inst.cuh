// Kernel instantiation and launch for one operand kind; included once by each
// tg_inst_<kind>.cu so the three kinds compile in parallel.
#pragma once

#include <atomic>
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
    kernel<<<a.grid, C::NUM_THREADS, C::SMEM_BYTES, a.stream>>>(a.map_a, a.map_b, a.p);
    return cudaGetLastError();
}

template <Kind KD>
static cudaError_t launch_kind(const LaunchArgs &a) {
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
