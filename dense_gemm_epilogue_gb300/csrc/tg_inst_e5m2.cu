// E5M2 kernel instantiations (compiled as their own translation unit).
#include "tg_inst.cuh"

namespace tg {
cudaError_t launch_e5m2(const LaunchArgs &a) { return launch_kind<Kind::E5M2>(a); }
}  // namespace tg
