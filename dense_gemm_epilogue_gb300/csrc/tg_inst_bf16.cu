// BF16 kernel instantiations (compiled as their own translation unit).
#include "tg_inst.cuh"

namespace tg {
cudaError_t launch_bf16(const LaunchArgs &a) { return launch_kind<Kind::BF16>(a); }
}  // namespace tg
