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
// copy behind.  A second kernel, launched as one thread-block cluster, runs the
// time-out path of the one-item kernels' cluster q/k roll: every thread arrives
// on the cluster barrier first, then the wait gives up, the CTA reports and
// still waits on the cluster barrier before it returns.
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

constexpr int kSelftestCluster = 4;

// mode 3: the cluster q/k roll's time-out path in each of kSelftestCluster
// CTAs; out[1] |= 4 when a CTA's wait gave up.
__global__ void __launch_bounds__(64) kda_cluster_wait_selftest_kernel(unsigned long long limit_ns, int* out) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    kda::mbar_init(&bar, 1);  // one arrival expected; none ever comes
    kda::fence_mbar_init();
  }
  __syncthreads();
  kda::cluster_arrive_release();  // where the verify kernel arrives: before any wait of its own
  const bool ok = kda::mbar_wait_bounded(&bar, 0, limit_ns);
  if (__syncthreads_or(!ok)) {
    if (threadIdx.x == 0) {
      atomicOr(out + 1, 4);
      atomicOr(out, kda::kStatusTmaTimeout);
    }
    kda::cluster_wait_acquire();  // every thread of the cluster arrived above
    return;
  }
  kda::cluster_wait_acquire();
}

}  // namespace

extern "C" int kda_selftest_bounded_wait(int mode, long long limit_ns, int* status, kda_stream_t stream) {
  if (!status) return KDA_ERR_NULL;
  if (mode < 0 || mode > 3 || limit_ns < 0 || limit_ns > (long long)kda::kWaitLimitNs) return KDA_ERR_SHAPE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (mode == 3) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(kSelftestCluster);
    lc.blockDim = dim3(64);
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSelftestCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&lc, kda_cluster_wait_selftest_kernel,
                                             static_cast<unsigned long long>(limit_ns), status);
    if (e != cudaSuccess) return (int)e;
    return (int)cudaGetLastError();
  }
  kda_wait_selftest_kernel<<<1, 64, 0, st>>>(mode, static_cast<unsigned long long>(limit_ns), status);
  return (int)cudaGetLastError();
}
