// bf16-activation instantiations of the ws verify-decode kernel.
#include "kda_launch.cuh"

namespace kda {
int launch_ws_bf16(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, cudaStream_t st) {
  return launch_ws_dispatch<__nv_bfloat16>(tmap, p, cfg, st);
}
}  // namespace kda
