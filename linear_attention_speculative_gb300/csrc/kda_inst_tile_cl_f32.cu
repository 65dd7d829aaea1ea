// f32-activation instantiations of the tile verify-decode kernel with the
// cluster q/k roll.
#include "kda_launch.cuh"

namespace kda {
int launch_tile_cluster_f32(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, cudaStream_t st) {
  return launch_tile_cluster_dispatch<float>(tmap, p, cfg, st);
}
}  // namespace kda
