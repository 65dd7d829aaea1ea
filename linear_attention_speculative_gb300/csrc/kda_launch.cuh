// kda_launch.cuh -- host-side launch of one kernel instantiation.  Each
// (activation type, kernel) pair is instantiated in its own translation unit
// (kda_inst_*.cu) so that they compile in parallel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "kda_kernel.cuh"

namespace kda {

struct LaunchCfg {
  int K;        // 32, 64, 128 or 256
  int warps;    // tile kernel: warps per CTA; pipelined kernel: consumer warps
  bool pipe;    // persistent warp-specialised (pipelined) kernel
  bool decode;  // tile kernel without snapshots, final state written in place
  bool sms;     // tile kernel with the state kept in shared memory
  bool split;   // split variant: prep kernel, then the tile kernel reading its stages
  int grid;     // CTAs
  size_t smem;  // dynamic shared memory bytes
};

// Launch the instantiation that matches `cfg`; returns a cudaError_t value,
// or -1 when no instantiation matches.
int launch_tile_bf16(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, cudaStream_t st);
int launch_tile_f32(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, cudaStream_t st);
int launch_pipe_bf16(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, cudaStream_t st);
int launch_pipe_f32(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, cudaStream_t st);
// The split variant: the prep kernel (grid N * H) and, as its programmatic
// dependent, the recurrence kernel (grid cfg.grid) on the same stream.
int launch_split_bf16(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, size_t prep_smem,
                      cudaStream_t st);
int launch_split_f32(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, size_t prep_smem,
                     cudaStream_t st);
// A one-item-per-CTA launch with p.qk_cluster > 1: the cluster-roll
// instantiations (kda_inst_tile_cl_*.cu; 4 or 8 warps, state in registers).
// A decode launch whose q/k conv_state needs no counter (one reader per
// group, or the separate roll kernel): the counter-free decode instantiations
// (kda_inst_tile_dec_*.cu).
int launch_tile_decode_bf16(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, cudaStream_t st);
int launch_tile_decode_f32(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, cudaStream_t st);
int launch_tile_cluster_bf16(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, cudaStream_t st);
int launch_tile_cluster_f32(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, cudaStream_t st);
// The q/k conv_state roll of a one-item-per-CTA launch run with
// p.qk_roll_kernel set (kda_roll.cu), on the same stream after it.
int launch_qk_roll(const Params& p, int K, bool bf16, cudaStream_t st);

// Launch as a programmatic dependent of the stream's previous kernel: the
// grid may be scheduled while that kernel's last CTAs run, and waits for it
// (griddepcontrol.wait) before its first global access.
inline void set_programmatic(cudaLaunchAttribute& a) {
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
}

// Opt a kernel in to large dynamic shared memory once per device.
template <typename Fn>
int configure_once(Fn fn, unsigned long long* configured) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return static_cast<int>(e);
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(__atomic_load_n(configured, __ATOMIC_ACQUIRE) & bit)) {
    int max_optin = 0;
    e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return static_cast<int>(e);
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_optin);
    if (e != cudaSuccess) return static_cast<int>(e);
    __atomic_fetch_or(configured, bit, __ATOMIC_RELEASE);
  }
  return 0;
}

template <typename Act, int K, int WARPS, bool DEC, bool SMS = false, int RM = kRollCounter>
int launch_tile_one(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, cudaStream_t st) {
  auto fn = kda_tile_kernel<Act, K, WARPS, DEC, SMS, false, RM>;
  static unsigned long long configured = 0;  // bit per device ordinal (< 64)
  int rc = configure_once(fn, &configured);
  if (rc) return rc;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)cfg.grid);
  lc.blockDim = dim3(WARPS * 32);
  lc.dynamicSmemBytes = cfg.smem;
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  set_programmatic(attr[0]);
  lc.attrs = attr;
  lc.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&lc, fn, tmap, p);
  if (e != cudaSuccess) return static_cast<int>(e);
  return static_cast<int>(cudaGetLastError());
}

// The cluster-roll instantiation (state in registers, 4 or 8 warps): the
// items of one q/k group -- consecutive CTAs, the grid a whole number of
// groups -- as one cluster of p.qk_cluster CTAs.
template <typename Act, int K, int WARPS, bool DEC>
int launch_tile_cluster_one(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, cudaStream_t st) {
  auto fn = kda_tile_kernel<Act, K, WARPS, DEC, false, false, kRollCluster>;
  static unsigned long long configured = 0;
  int rc = configure_once(fn, &configured);
  if (rc) return rc;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)cfg.grid);
  lc.blockDim = dim3(WARPS * 32);
  lc.dynamicSmemBytes = cfg.smem;
  lc.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.qk_cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  set_programmatic(attr[1]);
  lc.attrs = attr;
  lc.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&lc, fn, tmap, p);
  if (e != cudaSuccess) return static_cast<int>(e);
  return static_cast<int>(cudaGetLastError());
}

template <typename Act>
int launch_tile_cluster_dispatch(const CUtensorMap& tmap, const Params& p, const LaunchCfg& c, cudaStream_t st) {
  if (c.sms || p.qk_cluster < 2 || c.grid % p.qk_cluster != 0) return -1;
#define KDA_CASE(KK, WW)                                                              \
  if (c.K == KK && c.warps == WW)                                                     \
    return c.decode ? launch_tile_cluster_one<Act, KK, WW, true>(tmap, p, c, st)       \
                    : launch_tile_cluster_one<Act, KK, WW, false>(tmap, p, c, st);
#define KDA_CASES_K(KK) KDA_CASE(KK, 4) KDA_CASE(KK, 8)
  KDA_CASES_K(32)
  KDA_CASES_K(64)
  KDA_CASES_K(128)
  KDA_CASES_K(256)
#undef KDA_CASES_K
#undef KDA_CASE
  return -1;
}

template <typename Act, int K, int CW>
int launch_pipe_one(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, cudaStream_t st) {
  auto fn = kda_pipe_kernel<Act, K, CW>;
  static unsigned long long configured = 0;
  int rc = configure_once(fn, &configured);
  if (rc) return rc;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)cfg.grid);
  lc.blockDim = dim3(pipe_threads(CW));
  lc.dynamicSmemBytes = cfg.smem;
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  set_programmatic(attr[0]);
  lc.attrs = attr;
  lc.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&lc, fn, tmap, p);
  if (e != cudaSuccess) return static_cast<int>(e);
  return static_cast<int>(cudaGetLastError());
}

template <typename Act>
int launch_tile_dispatch(const CUtensorMap& tmap, const Params& p, const LaunchCfg& c, cudaStream_t st) {
#define KDA_CASE(KK, WW)                                                         \
  if (c.K == KK && c.warps == WW && !c.sms)                                       \
    return c.decode ? launch_tile_one<Act, KK, WW, true>(tmap, p, c, st)          \
                    : launch_tile_one<Act, KK, WW, false>(tmap, p, c, st);
#define KDA_CASE_SMS(KK, WW)                                                     \
  if (c.K == KK && c.warps == WW && c.sms)                                        \
    return c.decode ? launch_tile_one<Act, KK, WW, true, true>(tmap, p, c, st)    \
                    : launch_tile_one<Act, KK, WW, false, true>(tmap, p, c, st);
#define KDA_CASES_K(KK) KDA_CASE(KK, 1) KDA_CASE(KK, 2) KDA_CASE(KK, 4) KDA_CASE(KK, 8) \
  KDA_CASE_SMS(KK, 4) KDA_CASE_SMS(KK, 8)
  KDA_CASES_K(32)
  KDA_CASES_K(64)
  KDA_CASES_K(128)
  KDA_CASE(256, 2) KDA_CASE(256, 4) KDA_CASE(256, 8)
  KDA_CASE_SMS(256, 4)
  KDA_CASE_SMS(256, 8)
#undef KDA_CASES_K
#undef KDA_CASE_SMS
#undef KDA_CASE
  return -1;
}

// The decode instantiations without the arrival counter (kRollNone), for
// decode launches with one reader per q/k group or the separate roll kernel.
template <typename Act>
int launch_tile_decode_dispatch(const CUtensorMap& tmap, const Params& p, const LaunchCfg& c, cudaStream_t st) {
  if (!c.decode) return -1;
#define KDA_CASE(KK, WW)                                                                 \
  if (c.K == KK && c.warps == WW && !c.sms)                                               \
    return launch_tile_one<Act, KK, WW, true, false, kRollNone>(tmap, p, c, st);
#define KDA_CASE_SMS(KK, WW)                                                             \
  if (c.K == KK && c.warps == WW && c.sms)                                                \
    return launch_tile_one<Act, KK, WW, true, true, kRollNone>(tmap, p, c, st);
#define KDA_CASES_K(KK) KDA_CASE(KK, 1) KDA_CASE(KK, 2) KDA_CASE(KK, 4) KDA_CASE(KK, 8) \
  KDA_CASE_SMS(KK, 4) KDA_CASE_SMS(KK, 8)
  KDA_CASES_K(32)
  KDA_CASES_K(64)
  KDA_CASES_K(128)
  KDA_CASE(256, 2) KDA_CASE(256, 4) KDA_CASE(256, 8)
  KDA_CASE_SMS(256, 4)
  KDA_CASE_SMS(256, 8)
#undef KDA_CASES_K
#undef KDA_CASE_SMS
#undef KDA_CASE
  return -1;
}

template <typename Act, int K, int WARPS>
int launch_split_one(const CUtensorMap& tmap, const Params& p, const LaunchCfg& cfg, size_t prep_smem,
                     cudaStream_t st) {
  constexpr int BV = WARPS * warp_cols(K);
  auto prep = kda_prep_kernel<Act, K, BV>;
  auto rec = kda_tile_kernel<Act, K, WARPS, false, false, true, kRollCounter>;
  static unsigned long long configured_prep = 0, configured_rec = 0;
  int rc = configure_once(prep, &configured_prep);
  if (!rc) rc = configure_once(rec, &configured_rec);
  if (rc) return rc;
  cudaLaunchConfig_t pc = {};
  pc.gridDim = dim3((unsigned)(p.N * p.H));
  pc.blockDim = dim3(kPrepThreads);
  pc.dynamicSmemBytes = prep_smem;
  pc.stream = st;
  cudaLaunchAttribute pattr[1];
  set_programmatic(pattr[0]);
  pc.attrs = pattr;
  pc.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&pc, prep, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return static_cast<int>(e);
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)cfg.grid);
  lc.blockDim = dim3(WARPS * 32);
  lc.dynamicSmemBytes = cfg.smem;
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  set_programmatic(attr[0]);
  lc.attrs = attr;
  lc.numAttrs = 1;
  e = cudaLaunchKernelEx(&lc, rec, tmap, p);
  if (e != cudaSuccess) return static_cast<int>(e);
  return static_cast<int>(cudaGetLastError());
}

template <typename Act>
int launch_split_dispatch(const CUtensorMap& tmap, const Params& p, const LaunchCfg& c, size_t prep_smem,
                          cudaStream_t st) {
#define KDA_CASE(KK, WW) \
  if (c.K == KK && c.warps == WW) return launch_split_one<Act, KK, WW>(tmap, p, c, prep_smem, st);
#define KDA_CASES_K(KK) KDA_CASE(KK, 2) KDA_CASE(KK, 4) KDA_CASE(KK, 8)
  KDA_CASES_K(32)
  KDA_CASES_K(64)
  KDA_CASES_K(128)
#undef KDA_CASES_K
#undef KDA_CASE
  return -1;
}

template <typename Act>
int launch_pipe_dispatch(const CUtensorMap& tmap, const Params& p, const LaunchCfg& c, cudaStream_t st) {
#define KDA_CASE(KK, WW) \
  if (c.K == KK && c.warps == WW) return launch_pipe_one<Act, KK, WW>(tmap, p, c, st);
#define KDA_CASES_K(KK) KDA_CASE(KK, 4) KDA_CASE(KK, 8)
  KDA_CASES_K(32)
  KDA_CASES_K(64)
  KDA_CASES_K(128)
#undef KDA_CASES_K
#undef KDA_CASE
  return -1;
}

}  // namespace kda
