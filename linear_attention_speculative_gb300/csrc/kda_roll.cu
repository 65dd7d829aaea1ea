// kda_roll.cu -- the q/k conv_state roll as its own kernel
// ("[KDA] Fuse causal conv1d into MTP verify decode", cuLA pull request 107:
// conv_state is rolled in place to the last W-1 raw inputs of every channel).
//
// In the one-item-per-CTA verify kernels the q/k channels of group (n, h)
// are read by G * (V / BV) items.  None of them may overwrite that group's
// conv_state while another one may still read it, so when there are several
// readers the verify kernel leaves those channels alone and this kernel,
// launched right after it on the same stream, rolls them:
//     conv_state[slot(n), c, j] <- x_ext_c[T + j],  j = 0..2,
// for every q/k channel c, with x_ext_c = [conv_state[slot(n), c, :] ||
// mixed_qkv[n, :, c]] as the verify kernel saw it.  Stream order is the only
// synchronisation; the verify kernel needs no arrival counters for it.  The
// launch is a programmatic dependent of the verify kernel: its CTAs may be
// scheduled once every verify CTA has passed its own wait for the kernel
// before it (so whatever that kernel wrote is visible here too).  A thread
// first loads what it needs -- the new tokens, and for T < 3 the old q/k
// window, none of which the verify kernel writes -- and only then waits
// (griddepcontrol.wait, a hardware dependency wait) until the verify grid has
// completed, every read of the old window included, before it stores: the
// launch and the loads overlap the verify kernel's last wave.
//
// One thread per 16-byte vector of channels (8 bf16 / 4 fp32): it reads the
// vector's 3 old values per channel when T < 3 and the last min(T, 3) token
// rows of mixed_qkv, and writes the 48 bytes of the new window.  Sequences
// the verify kernel skipped (padding or out-of-range slots) are skipped here.
#include "kda_launch.cuh"

namespace kda {

namespace {

constexpr int kRollThreads = 256;

template <typename Act>
__global__ void __launch_bounds__(kRollThreads) kda_qk_roll_kernel(const Params p, int K) {
  using AT = ActT<Act>;
  using Raw = typename AT::Raw;
  constexpr int VEC = AT::VEC;
  const int per_seq = 2 * p.H * K / VEC;  // q/k channel vectors of one sequence
  const long long g = (long long)blockIdx.x * kRollThreads + threadIdx.x;
  if (g >= (long long)p.N * per_seq) return;
  const int n = static_cast<int>(g / per_seq);
  const int c = static_cast<int>(g - (long long)n * per_seq) * VEC;  // q then k channels
  const Item it = decode_item(p, (long long)n * p.HV * p.nvt);     // the sequence's first item
  if (it.skip) return;
  const int T = p.T;
  char* cp = reinterpret_cast<char*>(static_cast<Act*>(p.conv_state) +
                                     ((size_t)it.cs_row * p.dim + c) * (kConvW - 1));
  Raw old[3 * VEC] = {};
  if (T < kConvW - 1) {
#pragma unroll
    for (int m = 0; m < 3; ++m) AT::unpack(ld_rw_16(cp + 16 * m), old + m * VEC);
  }
  const Act* x = static_cast<const Act*>(p.mixed_qkv) + (size_t)n * T * p.dim + c;
  Raw r[3 * VEC];
#pragma unroll
  for (int j = 0; j < kConvW - 1; ++j) {
    const int idx = T + j;  // position in x_ext
    Raw xv[VEC];
    if (idx >= kConvW - 1) {
      AT::unpack(ld_ro_16(x + (size_t)(idx - (kConvW - 1)) * p.dim), xv);
    } else {
      select_state<Raw, VEC>(old, idx, xv);
    }
#pragma unroll
    for (int e = 0; e < VEC; ++e) r[e * (kConvW - 1) + j] = xv[e];
  }
  // the verify grid has completed (its reads of the old window too)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the next call's verify kernel may be scheduled as this one ends
  asm volatile("griddepcontrol.launch_dependents;");
#pragma unroll
  for (int m = 0; m < 3; ++m) st_16(cp + 16 * m, AT::pack(r + m * VEC));
}

}  // namespace

int launch_qk_roll(const Params& p, int K, bool bf16, cudaStream_t st) {
  const int vec = bf16 ? 8 : 4;
  const long long threads = (long long)p.N * (2LL * p.H * K / vec);
  if (threads == 0) return 0;
  const long long blocks = (threads + kRollThreads - 1) / kRollThreads;
  if (blocks > 0x7fffffffLL) return static_cast<int>(cudaErrorInvalidConfiguration);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kRollThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = bf16 ? cudaLaunchKernelEx(&cfg, kda_qk_roll_kernel<__nv_bfloat16>, p, K)
                             : cudaLaunchKernelEx(&cfg, kda_qk_roll_kernel<float>, p, K);
  if (e != cudaSuccess) return static_cast<int>(e);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace kda
