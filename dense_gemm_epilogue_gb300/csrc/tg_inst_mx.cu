// Block-scaled 8-bit / packed 4-bit float kernel instantiations and their launch (CTA-pair
// clusters, grid clamped to the pairs the device holds at once).
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include "tg_launch.h"

namespace tg {

template <Kind KD, int BN, bool PLAIN>
static cudaError_t launch_mx_one(const LaunchArgs &a) {
    using C = MxConfig<KD, BN>;
    auto kernel = tg_gemm_mx_kernel<KD, BN, PLAIN>;
    static std::atomic<uint64_t> configured{0};
    static int max_clusters[64] = {0};
    const uint64_t bit = (a.device >= 0 && a.device < 64) ? (1ull << a.device) : 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(C::threads(PLAIN), 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        int n = 0;
        cfg.gridDim = dim3(2, 1, 1);
        e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        if (bit) max_clusters[a.device] = n;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    int grid = a.grid - a.grid % 2;
    const int cap = bit ? 2 * max_clusters[a.device] : grid;
    if (grid > cap) grid = cap;
    if (grid < 2) grid = 2;
    cfg.gridDim = dim3(grid, 1, 1);
    if (std::getenv("TG_LOG"))
        std::fprintf(stderr, "tg_gemm_mx: BN=%d stages=%d grid=%d (planned %d) plain=%d\n", BN,
                     C::STAGES, grid, a.grid, PLAIN ? 1 : 0);
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, a.map_a, a.map_b, a.map_sfa, a.map_sfb, a.p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <Kind KD>
static cudaError_t launch_mx_kind(const LaunchArgs &a) {
    if (a.plain_loads) {
        if (a.block_n == 256) return launch_mx_one<KD, 256, true>(a);
        if (a.block_n == 128) return launch_mx_one<KD, 128, true>(a);
    } else {
        if (a.block_n == 256) return launch_mx_one<KD, 256, false>(a);
        if (a.block_n == 128) return launch_mx_one<KD, 128, false>(a);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_mx(const LaunchArgs &a, Kind kind) {
    if (kind == Kind::E4M3) return launch_mx_kind<Kind::E4M3>(a);
    if (kind == Kind::E5M2) return launch_mx_kind<Kind::E5M2>(a);
    if (kind == Kind::E2M1) return launch_mx_kind<Kind::E2M1>(a);
    if (kind == Kind::NVF4) return launch_mx_kind<Kind::NVF4>(a);
    return cudaErrorInvalidValue;
}

template <Kind KD>
static void mx_numbers(int block_n, bool plain, int *stages, int *smem, int *threads, int *tmem) {
    if (block_n == 256) {
        using C = MxConfig<KD, 256>;
        *stages = C::STAGES; *smem = C::SMEM_BYTES; *threads = C::threads(plain); *tmem = C::TMEM_COLS;
    } else if (block_n == 128) {
        using C = MxConfig<KD, 128>;
        *stages = C::STAGES; *smem = C::SMEM_BYTES; *threads = C::threads(plain); *tmem = C::TMEM_COLS;
    } else {
        *stages = *smem = *threads = *tmem = 0;
    }
}

void mx_config_numbers(Kind kind, int block_n, bool plain, int *stages, int *smem, int *threads,
                       int *tmem) {
    if (kind == Kind::E2M1) mx_numbers<Kind::E2M1>(block_n, plain, stages, smem, threads, tmem);
    else if (kind == Kind::NVF4) mx_numbers<Kind::NVF4>(block_n, plain, stages, smem, threads, tmem);
    else mx_numbers<Kind::E4M3>(block_n, plain, stages, smem, threads, tmem);
}

}  // namespace tg
