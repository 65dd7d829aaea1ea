// f32-activation instantiations of the pipelined (persistent, warp-specialised)
// verify-decode kernel.
#include "kda_launch.cuh"

namespace kda {
int launch_pipe_f32(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, cudaStream_t st) {
  return launch_pipe_dispatch<float>(tmap, p, cfg, st);
}
}  // namespace kda
