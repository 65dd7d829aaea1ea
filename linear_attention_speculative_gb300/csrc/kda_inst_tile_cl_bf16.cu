// bf16-activation instantiations of the tile verify-decode kernel with the
// cluster q/k roll.
#include "kda_launch.cuh"

namespace kda {
int launch_tile_cluster_bf16(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, cudaStream_t st) {
  return launch_tile_cluster_dispatch<__nv_bfloat16>(tmap, p, cfg, st);
}
}  // namespace kda
