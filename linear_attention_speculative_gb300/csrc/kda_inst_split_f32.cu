// f32-activation instantiations of the split variant: the prep kernel and the
// recurrence kernel that reads its stages.
#include "kda_launch.cuh"

namespace kda {
int launch_split_f32(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, size_t prep_smem,
                      cudaStream_t st) {
  return launch_split_dispatch<float>(tmap, p, cfg, prep_smem, st);
}
}  // namespace kda
