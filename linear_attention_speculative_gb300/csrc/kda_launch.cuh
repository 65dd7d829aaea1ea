// kda_launch.cuh -- host-side launch of one kernel instantiation.  Each
// activation type is instantiated in its own translation unit
// (kda_inst_bf16.cu, kda_inst_f32.cu) so the two compile in parallel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "kda_kernel.cuh"

namespace kda {

struct LaunchCfg {
  int K;        // 32, 64 or 128
  int warps;    // warps per CTA; the v-tile is 16 * warps columns
  bool persist; // persistent CTAs with next-tile prefetch
  int grid;     // CTAs
  size_t smem;  // dynamic shared memory bytes
};

// Launch the instantiation that matches `cfg`; returns a cudaError_t value,
// or -1 when no instantiation matches.
int launch_bf16(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, cudaStream_t st);
int launch_f32(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, cudaStream_t st);

template <typename Act, int K, int WARPS, bool PERSIST>
int launch_one(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, cudaStream_t st) {
  auto fn = kda_verify_kernel<Act, K, WARPS, PERSIST>;
  // Opt in to large dynamic shared memory once per device.
  static unsigned long long configured = 0;  // bit per device ordinal (< 64)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return static_cast<int>(e);
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & bit)) {
    int max_optin = 0;
    e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return static_cast<int>(e);
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_optin);
    if (e != cudaSuccess) return static_cast<int>(e);
    __atomic_fetch_or(&configured, bit, __ATOMIC_RELEASE);
  }
  fn<<<cfg.grid, WARPS * 32, cfg.smem, st>>>(tmap, p);
  return static_cast<int>(cudaGetLastError());
}

template <typename Act>
int launch_dispatch(const CUtensorMap& tmap, const Params& p, const LaunchCfg& c, cudaStream_t st) {
#define KDA_CASE(KK, WW, PP)                                      \
  if (c.K == KK && c.warps == WW && c.persist == PP)              \
    return launch_one<Act, KK, WW, PP>(tmap, p, c, st);
#define KDA_CASES_K(KK)                                           \
  KDA_CASE(KK, 1, false) KDA_CASE(KK, 2, false) KDA_CASE(KK, 4, false) \
  KDA_CASE(KK, 8, false) KDA_CASE(KK, 2, true) KDA_CASE(KK, 4, true)   \
  KDA_CASE(KK, 8, true)
  KDA_CASES_K(32)
  KDA_CASES_K(64)
  KDA_CASES_K(128)
#undef KDA_CASES_K
#undef KDA_CASE
  return -1;
}

}  // namespace kda
