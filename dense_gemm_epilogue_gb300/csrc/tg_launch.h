// Internal interface between the host front end (tg_gemm.cu) and the kernel
// instantiations (one translation unit per operand kind, compiled in parallel).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include "tg_kernel.cuh"

namespace tg {

struct LaunchArgs {
    GemmParams p;
    CUtensorMap map_a;   // A-role operand (unused by the plain-load producer)
    CUtensorMap map_b;   // B-role operand
    int block_n;         // 64, 128 or 256
    bool plain_loads;    // plain bounds-checked loads instead of TMA
    int grid;            // persistent CTAs
    int device;          // current device ordinal (for the per-device attribute cache)
    cudaStream_t stream;
};

cudaError_t launch_bf16(const LaunchArgs &a);
cudaError_t launch_fp16(const LaunchArgs &a);
cudaError_t launch_tf32(const LaunchArgs &a);

}  // namespace tg
