// f32-activation instantiations of the ws verify-decode kernel.
#include "kda_launch.cuh"

namespace kda {
int launch_ws_f32(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, cudaStream_t st) {
  return launch_ws_dispatch<float>(tmap, p, cfg, st);
}
}  // namespace kda
