// E4M3 kernel instantiations (compiled as their own translation unit).
#include "tg_inst.cuh"

namespace tg {
cudaError_t launch_e4m3(const LaunchArgs &a) { return launch_kind<Kind::E4M3>(a); }
}  // namespace tg
