// f32-activation instantiations of the tile decode kernel without the arrival
// counter.
#include "kda_launch.cuh"

namespace kda {
int launch_tile_decode_f32(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, cudaStream_t st) {
  return launch_tile_decode_dispatch<float>(tmap, p, cfg, st);
}
}  // namespace kda
