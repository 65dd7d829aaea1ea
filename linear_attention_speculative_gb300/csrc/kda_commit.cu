// kda_commit.cu -- kda_commit: accept the first acc[n] verified tokens of
// every sequence ("[KDA] Fuse causal conv1d into MTP verify decode", cuLA pull
// request 107: the verify writes per-token state and conv-window snapshots
// "for rollback"; this is that rollback / commit step).
//
// For each sequence n with 1 <= acc[n] <= T:
//     S[n]          <- inter_ssm[n, acc[n]-1]        (fp32, HV x K x V)
//     conv_state[n] <- conv_snapshots[n, acc[n]-1]   (act, dim x 3)
// A pure HBM copy of 16-byte vectors over a non-persistent grid: each CTA
// copies one 16 KiB chunk of one sequence's state + conv window (the sequence
// and chunk come from the block index, so no per-element division), every
// thread issuing all four of its streaming loads before its four stores so
// that 64 bytes per thread are in flight.  Sequences whose count is out of
// range are left untouched and reported in the status word.  The launch is a
// programmatic dependent of the stream's previous kernel: its CTAs may start
// while that kernel ends and wait for it before any global access.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "kda_device.cuh"
#include "../../include/kda_verify.h"

namespace {

constexpr int kCommitThreads = 256;
constexpr int kCommitUnroll = 4;

struct CommitParams {
  const int32_t* acc;
  const int32_t* idx_state;  // optional pool slots (NULL: slot = n)
  const int32_t* idx_conv;
  const int32_t* idx_inter;
  long long pool_state, pool_conv, pool_inter;
  const float* inter_ssm;
  const unsigned char* snaps;
  float* S;
  unsigned char* conv_state;
  int* status;
  long long state_vecs;  // 16-byte vectors of one sequence's state (HV*K*V/4)
  long long conv_vecs;   // 16-byte vectors of one sequence's conv window
  int chunks;            // CTAs per sequence: ceil((state_vecs + conv_vecs) / kCommitChunk)
  int T;
};

constexpr int kCommitChunk = kCommitThreads * kCommitUnroll;  // vectors per CTA

__global__ void __launch_bounds__(kCommitThreads) kda_commit_kernel(const CommitParams p) {
  // launched as a programmatic dependent of the stream's previous kernel (the
  // verify, as a rule): nothing global is touched before it has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const long long n = blockIdx.x / p.chunks;
  const long long r0 = (long long)(blockIdx.x - n * p.chunks) * kCommitChunk + threadIdx.x;
  const long long ss = p.idx_state ? __ldg(p.idx_state + n) : n;
  const long long sc = p.idx_conv ? __ldg(p.idx_conv + n) : n;
  const long long si = p.idx_inter ? __ldg(p.idx_inter + n) : n;
  if (ss < 0 || sc < 0 || si < 0) return;  // padding sequence
  const bool first = r0 == 0;               // one report per sequence
  if (ss >= p.pool_state || sc >= p.pool_conv || si >= p.pool_inter) {
    if (first && p.status) atomicOr(p.status, KDA_STATUS_BAD_INDEX);
    return;
  }
  const int a = __ldg(p.acc + n);
  if (a < 1 || a > p.T) {
    if (first && p.status) atomicOr(p.status, KDA_STATUS_BAD_ACCEPT);
    return;
  }
  const long long per_seq = p.state_vecs + p.conv_vecs;
  const uint4* ssrc = reinterpret_cast<const uint4*>(p.inter_ssm) + (si * p.T + (a - 1)) * p.state_vecs;
  uint4* sdst = reinterpret_cast<uint4*>(p.S) + ss * p.state_vecs;
  const uint4* csrc = reinterpret_cast<const uint4*>(p.snaps) + (si * p.T + (a - 1)) * p.conv_vecs;
  uint4* cdst = reinterpret_cast<uint4*>(p.conv_state) + sc * p.conv_vecs;
  uint4 v[kCommitUnroll] = {};
#pragma unroll
  for (int u = 0; u < kCommitUnroll; ++u) {
    const long long r = r0 + (long long)u * kCommitThreads;
    if (r < p.state_vecs) v[u] = __ldcs(ssrc + r);
    else if (r < per_seq) v[u] = __ldcs(csrc + (r - p.state_vecs));
  }
#pragma unroll
  for (int u = 0; u < kCommitUnroll; ++u) {
    const long long r = r0 + (long long)u * kCommitThreads;
    if (r < p.state_vecs) __stcs(sdst + r, v[u]);
    else if (r < per_seq) __stcs(cdst + (r - p.state_vecs), v[u]);
  }
}

bool overlap(uintptr_t a, size_t na, uintptr_t b, size_t nb) {
  return na && nb && a < b + nb && b < a + na;
}

}  // namespace

extern "C" int kda_commit_indexed(const kda_shape* s, const kda_state_indices* idx,
                                  const int32_t* accepted, const float* inter_ssm,
                                  const void* conv_snapshots, float* S, void* conv_state,
                                  int* status, kda_stream_t stream) {
  if (!s) return KDA_ERR_NULL;
  if (s->act != KDA_F32 && s->act != KDA_BF16) return KDA_ERR_DTYPE;
  if (s->N < 0 || s->T < 1 || s->T > KDA_MAX_T || s->H < 1 || s->HV < s->H ||
      s->HV % s->H != 0 || s->W != 4 || (s->K != 32 && s->K != 64 && s->K != 128 && s->K != 256) ||
      (s->V != 32 && s->V != 64 && s->V != 128 && s->V != 256))
    return KDA_ERR_SHAPE;
  if (s->N == 0) return KDA_OK;
  if (!accepted || !inter_ssm || !conv_snapshots || !S || !conv_state) return KDA_ERR_NULL;
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!al16(inter_ssm) || !al16(conv_snapshots) || !al16(S) || !al16(conv_state) ||
      (reinterpret_cast<uintptr_t>(accepted) & 3u) || (reinterpret_cast<uintptr_t>(status) & 3u))
    return KDA_ERR_MISALIGNED;
  const size_t ab = s->act == KDA_F32 ? 4 : 2;
  const size_t N = s->N, T = s->T, HV = s->HV, K = s->K, V = s->V;
  const size_t dim = 2 * (size_t)s->H * K + HV * V;
  size_t ps = N, pc = N, pi = N;
  const int32_t *is = nullptr, *ic = nullptr, *ii = nullptr;
  if (idx) {
    if (idx->cache_indices) { if (idx->state_pool < 1) return KDA_ERR_SHAPE; is = idx->cache_indices; ps = idx->state_pool; }
    if (idx->conv_state_indices) { if (idx->conv_pool < 1) return KDA_ERR_SHAPE; ic = idx->conv_state_indices; pc = idx->conv_pool; }
    if (idx->intermediate_state_indices) { if (idx->inter_pool < 1) return KDA_ERR_SHAPE; ii = idx->intermediate_state_indices; pi = idx->inter_pool; }
    if ((reinterpret_cast<uintptr_t>(is) | reinterpret_cast<uintptr_t>(ic) | reinterpret_cast<uintptr_t>(ii)) & 3u)
      return KDA_ERR_MISALIGNED;
  }
  const uintptr_t in[6][2] = {{reinterpret_cast<uintptr_t>(accepted), N * 4},
                              {reinterpret_cast<uintptr_t>(inter_ssm), pi * T * HV * K * V * 4},
                              {reinterpret_cast<uintptr_t>(conv_snapshots), pi * T * dim * 3 * ab},
                              {reinterpret_cast<uintptr_t>(is), is ? N * 4 : 0},
                              {reinterpret_cast<uintptr_t>(ic), ic ? N * 4 : 0},
                              {reinterpret_cast<uintptr_t>(ii), ii ? N * 4 : 0}};
  const uintptr_t out[3][2] = {{reinterpret_cast<uintptr_t>(S), ps * HV * K * V * 4},
                               {reinterpret_cast<uintptr_t>(conv_state), pc * dim * 3 * ab},
                               {reinterpret_cast<uintptr_t>(status), status ? 4u : 0u}};
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 6; ++j)
      if (overlap(out[i][0], out[i][1], in[j][0], in[j][1])) return KDA_ERR_ALIAS;
    for (int j = 0; j < 3; ++j)
      if (j != i && overlap(out[i][0], out[i][1], out[j][0], out[j][1])) return KDA_ERR_ALIAS;
  }
  CommitParams p;
  p.acc = accepted;
  p.idx_state = is;
  p.idx_conv = ic;
  p.idx_inter = ii;
  p.pool_state = (long long)ps;
  p.pool_conv = (long long)pc;
  p.pool_inter = (long long)pi;
  p.inter_ssm = inter_ssm;
  p.snaps = static_cast<const unsigned char*>(conv_snapshots);
  p.S = S;
  p.conv_state = static_cast<unsigned char*>(conv_state);
  p.status = status;
  p.state_vecs = (long long)(HV * K * V / 4);
  p.conv_vecs = (long long)(dim * 3 * ab / 16);
  const long long chunks = (p.state_vecs + p.conv_vecs + kCommitChunk - 1) / kCommitChunk;
  p.T = s->T;
  const long long blocks = (long long)N * chunks;
  if (chunks > 0x7fffffffLL || blocks > 0x7fffffffLL) return KDA_ERR_SHAPE;
  p.chunks = (int)chunks;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)blocks);
  lc.blockDim = dim3(kCommitThreads);
  lc.dynamicSmemBytes = 0;
  lc.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&lc, kda_commit_kernel, p);
  if (e != cudaSuccess) return static_cast<int>(e);
  return static_cast<int>(cudaGetLastError());
}

extern "C" int kda_commit(const kda_shape* s, const int32_t* accepted, const float* inter_ssm,
                          const void* conv_snapshots, float* S, void* conv_state, int* status,
                          kda_stream_t stream) {
  return kda_commit_indexed(s, nullptr, accepted, inter_ssm, conv_snapshots, S, conv_state, status,
                            stream);
}
