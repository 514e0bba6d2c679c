// FP16 kernel instantiations (compiled as their own translation unit).
#include "tg_inst.cuh"

namespace tg {
cudaError_t launch_fp16(const LaunchArgs &a) { return launch_kind<Kind::FP16>(a); }
}  // namespace tg
