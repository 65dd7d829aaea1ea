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
// first call before any stream capture.  The address is kept per device
// together with the driver context it was looked up in; a call made in
// another context (after cudaDeviceReset, or under a context the caller made
// current) looks it up again.  Each call then clears the scratch it uses with
// cudaMemsetAsync on the caller's stream and launches the same kernels as
// kda_conv_verify.  No call allocates or frees memory.
//
// The kernels report a bounded wait that gave up, or a skipped sequence, in
// the status word of the scratch; kda_noalloc_read_status reads (and clears)
// it.  The next call clears it as well, so read it before that.
//
// Every call shares the one array: two calls whose kernels overlap on the GPU
// (different streams, or different host threads on the same device) race on
// the counters and the status word and can give wrong conv_state write-backs.
// Serialise them.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/kda_verify.h"

namespace {

constexpr size_t kNoallocScratchBytes = KDA_NOALLOC_MAX_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  CUcontext ctx;
  void* addr;
};
ScratchSlot g_scratch[kMaxDevices] = {};
std::mutex g_scratch_mutex;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry-point query (no link
// against the driver library).
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of the array in the current device's current context.
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return static_cast<int>(e);
  if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_DEVICE;
  CtxGetCurrentFn get = ctx_get_current();
  CUcontext ctx = nullptr;
  if (!get || get(&ctx) != CUDA_SUCCESS) return KDA_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!ctx || !g_scratch[dev].addr || g_scratch[dev].ctx != ctx) {
    void* p = nullptr;
    // also makes the runtime's context current when none was
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return static_cast<int>(e);
    if (!p) return KDA_ERR_DEVICE;
    if (!ctx && (get(&ctx) != CUDA_SUCCESS || !ctx)) return KDA_ERR_DEVICE;
    g_scratch[dev].ctx = ctx;
    g_scratch[dev].addr = p;
  }
  *out = g_scratch[dev].addr;
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
  // An empty batch launches nothing: the regular entry point checks the
  // shape and gate mode and returns without touching a workspace.
  if (s->N == 0)
    return kda_conv_verify(s, mixed_qkv, conv_w, conv_state, A_log, dt_bias, a, b, S0, gate_mode,
                           o, inter_ssm, conv_snapshots, nullptr, 0, stream);
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc) return rc;
  // The array keeps whatever the previous call left: start from zero.
  cudaError_t e = cudaMemsetAsync(scratch, 0, need, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return static_cast<int>(e);
  return kda_conv_verify(s, mixed_qkv, conv_w, conv_state, A_log, dt_bias, a, b, S0, gate_mode,
                         o, inter_ssm, conv_snapshots, scratch, kNoallocScratchBytes, stream);
}

extern "C" int kda_noalloc_read_status(const kda_shape* s, int* status, kda_stream_t stream) {
  if (!s || !status) return KDA_ERR_NULL;
  if (kda_workspace_bytes(s) > kNoallocScratchBytes) return KDA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc) return rc;
  return kda_read_status(s, scratch, status, stream);
}
