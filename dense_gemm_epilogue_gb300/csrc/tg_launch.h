// Internal interface between the host front end (tg_gemm.cu) and the kernel
// instantiations (one translation unit per operand kind, compiled in parallel).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include "tg_kernel.cuh"
#include "tg_kernel_pair.cuh"
#include "tg_kernel_mx.cuh"

namespace tg {

struct LaunchArgs {
    GemmParams p;
    CUtensorMap map_a;   // A-role operand (unused by the plain-load producer)
    CUtensorMap map_b;   // B-role operand
    CUtensorMap map_sfa; // block-scaled kernel: A-role scale atoms
    CUtensorMap map_sfb; // block-scaled kernel: B-role scale atoms
    int block_n;         // tile N: 64, 128 or 256 (single CTA); 128 or 256 (CTA pair)
    bool plain_loads;    // plain bounds-checked loads instead of TMA (single-CTA and block-scaled kernels)
    bool pair;           // CTA-pair kernel (cta_group::2 MMA)
    int mc;              // pair kernel: pairs per cluster (1, or 2 with A multicast)
    int grid;            // persistent CTAs (even for the pair kernel)
    int device;          // current device ordinal (for the per-device attribute cache)
    cudaStream_t stream;
};

cudaError_t launch_bf16(const LaunchArgs &a);
cudaError_t launch_fp16(const LaunchArgs &a);
cudaError_t launch_tf32(const LaunchArgs &a);
cudaError_t launch_e4m3(const LaunchArgs &a);
cudaError_t launch_e5m2(const LaunchArgs &a);
// Block-scaled 8-bit / packed 4-bit float kernel (CTA pairs, block_n 128 or 256).
cudaError_t launch_mx(const LaunchArgs &a, Kind kind);
// The K == 0 case (empty sums): D = out(epi(alpha * 0)) over `batch` M x N
// outputs, `stride_d` output elements apart, enqueued on `stream`.  One
// kernel launch; allocates nothing.
cudaError_t launch_fill_empty_sum(void *d, int64_t m, int64_t n, int64_t ldc, int64_t stride_d,
                                  int64_t batch, int out_fmt, float alpha, int relu,
                                  const EpiProgram &prog, int sms, cudaStream_t stream);
// Threads, shared memory, stages and tensor-memory columns of a block-scaled
// configuration (0 when the configuration does not exist).
void mx_config_numbers(Kind kind, int block_n, bool plain, int *stages, int *smem, int *threads,
                       int *tmem);

}  // namespace tg
