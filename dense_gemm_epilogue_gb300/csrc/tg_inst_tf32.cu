// TF32 kernel instantiations (compiled as their own translation unit).
#include "tg_inst.cuh"

namespace tg {
cudaError_t launch_tf32(const LaunchArgs &a) { return launch_kind<Kind::TF32>(a); }
}  // namespace tg
