// kda_noalloc.cu -- kda_conv_verify_noalloc: the verify decode for callers
// that cannot allocate device memory.
//
// The regular entry point asks the caller for a workspace (a status word and
// the q/k arrival counters that small launches use).  Some callers have no way to provide one: a
// plugin handed only its input and output buffers, a serving loop whose
// memory pool is frozen after start-up, or code that must not call
// cudaMalloc because it synchronises the device and can fail under a memory
// cap.  For them the scratch lives in a fixed array in this library's device
// image, sized at build time (kNoallocScratchBytes below); every GPU that
// loads the library holds that array until the process exits.
//
// Set-up: the first call on a device, with that device current, looks up the
// array's device address with cudaGetSymbolAddress (the array's name in host
// code is only a host-side stand-in, never a device address).  Make that
// first call before any stream capture.  Each call then clears the scratch
// it uses with cudaMemsetAsync on the caller's stream and launches the same
// kernels as kda_conv_verify.  No call allocates or frees memory.
//
// Every call shares the one array: two calls whose kernels overlap on the GPU
// (different streams, or different host threads on the same device) race on
// the counters and the status word and can give wrong conv_state write-backs.
// Serialise them.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/kda_verify.h"

namespace {

constexpr size_t kNoallocScratchBytes = KDA_NOALLOC_MAX_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mutex;

// Device address of the array on the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return static_cast<int>(e);
  if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return static_cast<int>(e);
    if (!p) return KDA_ERR_DEVICE;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return KDA_OK;
}

}  // namespace

extern "C" int kda_conv_verify_noalloc(const kda_shape* s, const void* mixed_qkv,
                                       const void* conv_w, void* conv_state,
                                       const float* A_log, const float* dt_bias, const void* a,
                                       const void* b, const float* S0, kda_gate_mode gate_mode,
                                       void* o, float* inter_ssm, void* conv_snapshots,
                                       kda_stream_t stream) {
  if (!s) return KDA_ERR_NULL;
  const size_t need = kda_workspace_bytes(s);
  if (need > kNoallocScratchBytes) return KDA_ERR_SCRATCH_LIMIT;
  if (s->N == 0) return KDA_OK;
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc) return rc;
  // The array keeps whatever the previous call left: start from zero.
  cudaError_t e = cudaMemsetAsync(scratch, 0, need, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return static_cast<int>(e);
  return kda_conv_verify(s, mixed_qkv, conv_w, conv_state, A_log, dt_bias, a, b, S0, gate_mode,
                         o, inter_ssm, conv_snapshots, scratch, kNoallocScratchBytes, stream);
}
