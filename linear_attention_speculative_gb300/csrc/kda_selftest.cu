// kda_selftest.cu -- the device-side bounded waits exercised without a fault.
//
// Every wait of the verify kernels is bounded: past its limit the waiting
// thread gives up, the kernel records KDA_STATUS_TMA_TIMEOUT in the status word
// and returns, and the CUDA context stays usable.  This one-CTA kernel runs the
// same wait helpers against an mbarrier that nothing ever arrives at, so the
// limit is reached on purpose: warp 0 in mbar_wait_bounded (the one-item
// kernels' wait, here with the caller's limit), warp 1 in pipe_wait (the
// pipelined kernel's wait: its fixed limit, or earlier when the group's abort
// flag is raised).  Nothing is in flight on the barrier, so giving up leaves no
// copy behind.
#include "kda_kernel.cuh"
#include "../../include/kda_verify.h"

namespace {

// mode 0: warp 0 waits (limit_ns); mode 1: warp 0 waits (limit_ns) and, when it
// gives up, raises the abort flag that ends warp 1's pipe_wait; mode 2: warp 1's
// pipe_wait alone, until its own limit.  out[0] |= KDA_STATUS_TMA_TIMEOUT when a
// wait gave up; out[1] |= 1 (mbar_wait_bounded gave up), 2 (pipe_wait did).
__global__ void __launch_bounds__(64) kda_wait_selftest_kernel(int mode, unsigned long long limit_ns,
                                                               int* out) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    kda::mbar_init(&bar, 1);  // one arrival expected; none ever comes
    abort_flag = 0;
    kda::fence_mbar_init();
  }
  __syncthreads();
  int mask = 0;
  if (warp == 0 && mode != 2) {
    if (!kda::mbar_wait_bounded(&bar, 0, limit_ns)) {
      mask |= 1;
      if (mode == 1 && lane == 0) *reinterpret_cast<volatile int*>(&abort_flag) = 1;
    }
  }
  if (warp == 1 && mode != 0) {
    if (!kda::pipe_wait(&bar, 0, &abort_flag)) mask |= 2;
  }
  if (lane == 0 && mask) {
    atomicOr(out + 1, mask);
    atomicOr(out, kda::kStatusTmaTimeout);
  }
}

}  // namespace

extern "C" int kda_selftest_bounded_wait(int mode, long long limit_ns, int* status, kda_stream_t stream) {
  if (!status) return KDA_ERR_NULL;
  if (mode < 0 || mode > 2 || limit_ns < 0 || limit_ns > (long long)kda::kWaitLimitNs) return KDA_ERR_SHAPE;
  kda_wait_selftest_kernel<<<1, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      mode, static_cast<unsigned long long>(limit_ns), status);
  return (int)cudaGetLastError();
}
