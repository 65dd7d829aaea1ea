// kda_kernel.cuh -- the fused causal-conv1d + KDA verify-decode kernel for
// sm_103a ("[KDA] Fuse causal conv1d into MTP verify decode", cuLA pull
// request 107).
//
// Work item: (sequence n, value head hv, v-tile vt) = a K x BV slice of one
// recurrent state.  A CTA of WARPS warps owns BV = 16 * WARPS columns.
//
//   producer  conv1d(W=4) + SiLU of the q/k channels of head h = hv / G and of
//             the tile's v channels for all T tokens, q/k L2 norm (q scaled by
//             K^-1/2), alpha = exp(g) and beta, staged in shared memory; the
//             raw conv windows are streamed out as snapshots.  All global
//             loads are 16-byte vectors.
//   state     the item's S0 slice arrives in shared memory by one 2-D TMA
//             tile load (mbarrier completion); in the persistent variant the
//             next item's tile is requested as soon as the current one has
//             moved to registers, so the load overlaps the recurrence.
//   consumer  every warp owns 16 columns; lane = (row group rg in 0..7,
//             column quad cg in 0..3) keeps rows [rg*K/8, (rg+1)*K/8) x 4
//             columns of S in registers.  Per token: decay + S^T k partial
//             sums, a 3-step xor butterfly across the row groups, the rank-1
//             update fused with the S^T q partial sums and the 16-byte
//             streaming store of the snapshot, a second butterfly, o.
//
// Both variants (one item per CTA, or persistent CTAs) run the same
// producer/consumer code with the same per-warp layout, hence the same
// floating-point operation order: their outputs are bit-identical.
//
// Shared q/k conv_state write-back: the q/k channels of group (n, h) are read
// by G * (V / BV) items.  Each item arrives on a per-group counter after its
// reads; the last arrival rolls the group's q/k conv_state and resets the
// counter to zero.  Nothing ever waits on another CTA.  v channels belong to
// exactly one item, which rolls them right after reading them.
#pragma once

#include "kda_device.cuh"

namespace kda {

struct Params {
  const void* mixed_qkv;  // act [N, T, dim]
  const void* conv_w;     // act [dim, 4]
  void* conv_state;       // act [N, dim, 3]
  const float* A_log;     // f32 [HV]
  const float* dt_bias;   // f32 [HV, K]
  const void* a;          // act [N, T, HV, K]
  const void* b;          // act [N, T, HV]
  void* o;                // act [N, T, HV, V]
  float* inter_ssm;       // f32 [N, T, HV, K, V]
  void* conv_snapshots;   // act [N, T, dim, 3]
  int* counters;          // [N * H]
  int* status;            // device status word
  long long num_items;    // N * HV * nvt
  int N, T, H, HV, V, dim, G, nvt;
  int gate_mode;          // 0 softplus, 1 safe
};

constexpr int kConvW = 4;
constexpr float kL2Eps = 1e-6f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__host__ __device__ constexpr int round4(int x) { return (x + 3) & ~3; }

// floats of one stage: q[T][K], k[T][K], alpha[T][K], v[T][BV], beta[round4(T)]
__host__ __device__ constexpr int stage_floats(int T, int K, int BV) {
  return 3 * T * K + T * BV + round4(T);
}

__host__ __device__ constexpr size_t smem_bytes(int T, int K, int BV, int nstage) {
  return 128 + sizeof(float) * (size_t)K * BV + sizeof(float) * (size_t)nstage * stage_floats(T, K, BV);
}

struct Item {
  int n, hv, h, vt;
  long long unit;  // n * HV + hv
};

__device__ __forceinline__ Item decode_item(const Params& p, long long item) {
  Item it;
  it.unit = item / p.nvt;
  it.vt = static_cast<int>(item - it.unit * p.nvt);
  it.n = static_cast<int>(it.unit / p.HV);
  it.hv = static_cast<int>(it.unit - (long long)it.n * p.HV);
  it.h = it.hv / p.G;
  return it;
}

// ---------------------------------------------------------------------------
// producer phase 1: conv + SiLU (q, k, v), gate, beta
// ---------------------------------------------------------------------------
template <typename Act, int K, int BV, int NT>
__device__ __forceinline__ void produce_phase1(const Params& p, const Item& it, float* sQ,
                                               float* sK, float* sA, float* sV, float* sB,
                                               int tid) {
  using AT = ActT<Act>;
  using Raw = typename AT::Raw;
  constexpr int VEC = AT::VEC;
  constexpr int NQ = K / VEC;   // channel vectors per q (or k) head
  constexpr int NVV = BV / VEC; // channel vectors of the v tile
  constexpr int NCONV = 2 * NQ + NVV;
  const int T = p.T;
  const int dim = p.dim;
  const int ntask_gate = T * NQ;
  const int ntask = NCONV + ntask_gate + T;
  // q/k snapshots are written once per group: by its first v-head, first tile
  const bool qk_snap_owner = (it.hv % p.G == 0) && (it.vt == 0);

  const Act* xq = static_cast<const Act*>(p.mixed_qkv) + (size_t)it.n * T * dim;
  Act* cs_base = static_cast<Act*>(p.conv_state) + (size_t)it.n * dim * (kConvW - 1);
  Act* snap_base = static_cast<Act*>(p.conv_snapshots) + (size_t)it.n * T * dim * (kConvW - 1);

  for (int task = tid; task < ntask; task += NT) {
    if (task < NCONV) {
      int c, kind, e0;
      if (task < NQ) {
        kind = 0; e0 = task * VEC; c = it.h * K + e0;
      } else if (task < 2 * NQ) {
        kind = 1; e0 = (task - NQ) * VEC; c = p.H * K + it.h * K + e0;
      } else {
        kind = 2; e0 = (task - 2 * NQ) * VEC; c = 2 * p.H * K + it.hv * p.V + it.vt * BV + e0;
      }
      // weights: VEC channels x 4 taps = 4 x 16 bytes
      float wf[VEC][kConvW];
      {
        const char* wp = reinterpret_cast<const char*>(static_cast<const Act*>(p.conv_w) +
                                                       (size_t)c * kConvW);
        Raw r[4 * VEC];
#pragma unroll
        for (int m = 0; m < 4; ++m) AT::unpack(ld_ro_16(wp + 16 * m), r + m * VEC);
#pragma unroll
        for (int e = 0; e < VEC; ++e)
#pragma unroll
          for (int j = 0; j < kConvW; ++j) wf[e][j] = AT::to_f(r[e * kConvW + j]);
      }
      // conv window: 3 state values (oldest first) + the current token
      Raw win[VEC][kConvW];
      Act* csp = cs_base + (size_t)c * (kConvW - 1);
      {
        Raw r[3 * VEC];
#pragma unroll
        for (int m = 0; m < 3; ++m)
          AT::unpack(ld_rw_16(reinterpret_cast<const char*>(csp) + 16 * m), r + m * VEC);
#pragma unroll
        for (int e = 0; e < VEC; ++e)
#pragma unroll
          for (int j = 0; j < kConvW - 1; ++j) win[e][j] = r[e * (kConvW - 1) + j];
      }
      const bool snap = (kind == 2) || qk_snap_owner;
      float* dst = kind == 0 ? sQ + e0 : (kind == 1 ? sK + e0 : sV + e0);
      const int dstride = kind == 2 ? BV : K;
      uint4 xnext = ld_ro_16(xq + c);
      for (int t = 0; t < T; ++t) {
        const uint4 xv = xnext;
        if (t + 1 < T) xnext = ld_ro_16(xq + (size_t)(t + 1) * dim + c);
        {
          Raw r[VEC];
          AT::unpack(xv, r);
#pragma unroll
          for (int e = 0; e < VEC; ++e) win[e][kConvW - 1] = r[e];
        }
        float y[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          float acc = __fmul_rn(wf[e][0], AT::to_f(win[e][0]));
#pragma unroll
          for (int j = 1; j < kConvW; ++j) acc = __fmaf_rn(wf[e][j], AT::to_f(win[e][j]), acc);
          y[e] = silu_f(acc);
        }
#pragma unroll
        for (int e = 0; e < VEC; e += 4)
          *reinterpret_cast<float4*>(dst + t * dstride + e) = make_float4(y[e], y[e + 1], y[e + 2], y[e + 3]);
        if (snap) {
          Raw r[3 * VEC];
#pragma unroll
          for (int e = 0; e < VEC; ++e)
#pragma unroll
            for (int j = 0; j < kConvW - 1; ++j) r[e * (kConvW - 1) + j] = win[e][j + 1];
          char* sp = reinterpret_cast<char*>(snap_base + ((size_t)t * dim + c) * (kConvW - 1));
#pragma unroll
          for (int m = 0; m < 3; ++m) st_16(sp + 16 * m, AT::pack(r + m * VEC));
        }
#pragma unroll
        for (int e = 0; e < VEC; ++e)
#pragma unroll
          for (int j = 0; j < kConvW - 1; ++j) win[e][j] = win[e][j + 1];
      }
      if (kind == 2) {
        // v channels are read by this item only: roll them in place now
        Raw r[3 * VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e)
#pragma unroll
          for (int j = 0; j < kConvW - 1; ++j) r[e * (kConvW - 1) + j] = win[e][j];
#pragma unroll
        for (int m = 0; m < 3; ++m) st_16(reinterpret_cast<char*>(csp) + 16 * m, AT::pack(r + m * VEC));
      }
    } else if (task < NCONV + ntask_gate) {
      const int g = task - NCONV;
      const int t = g / NQ;
      const int e0 = (g - t * NQ) * VEC;
      const Act* ap = static_cast<const Act*>(p.a) + (((size_t)it.n * T + t) * p.HV + it.hv) * K + e0;
      Raw r[VEC];
      AT::unpack(ld_ro_16(ap), r);
      float al[VEC];
      if (p.gate_mode == 0) {
        const float negA = -expf(__ldg(p.A_log + it.hv));
        const float* dtp = p.dt_bias + (size_t)it.hv * K + e0;
#pragma unroll
        for (int e = 0; e < VEC; e += 4) {
          const float4 d = __ldg(reinterpret_cast<const float4*>(dtp + e));
          const float dd[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float x = __fadd_rn(AT::to_f(r[e + j]), dd[j]);
            al[e + j] = expf(__fmul_rn(negA, softplus_f(x)));
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) al[e] = expf(fminf(AT::to_f(r[e]), 0.0f));
      }
#pragma unroll
      for (int e = 0; e < VEC; e += 4)
        *reinterpret_cast<float4*>(sA + t * K + e0 + e) = make_float4(al[e], al[e + 1], al[e + 2], al[e + 3]);
    } else {
      const int t = task - NCONV - ntask_gate;
      const Act* bp = static_cast<const Act*>(p.b) + ((size_t)it.n * T + t) * p.HV + it.hv;
      float bv;
      if constexpr (sizeof(Act) == 4) {
        bv = __ldg(reinterpret_cast<const float*>(bp));
      } else {
        bv = AT::to_f(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(bp))));
      }
      sB[t] = sigmoid_f(bv);
    }
  }
}

// ---------------------------------------------------------------------------
// producer phase 2: L2 norm of q and k per token (one warp per vector)
// ---------------------------------------------------------------------------
template <int K, int WARPS>
__device__ __forceinline__ void produce_phase2(int T, float* sQ, float* sK, int warp, int lane) {
  const float scale = rsqrtf(static_cast<float>(K));
  for (int r = warp; r < 2 * T; r += WARPS) {
    float* x = r < T ? sQ + r * K : sK + (r - T) * K;
    float xs[K / 32];
    float ss = 0.0f;
#pragma unroll
    for (int m = 0; m < K / 32; ++m) {
      xs[m] = x[lane + 32 * m];
      ss = __fmaf_rn(xs[m], xs[m], ss);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
    float inv = rsqrtf(__fadd_rn(ss, kL2Eps));
    if (r < T) inv = __fmul_rn(inv, scale);
#pragma unroll
    for (int m = 0; m < K / 32; ++m) x[lane + 32 * m] = __fmul_rn(xs[m], inv);
  }
}

// ---------------------------------------------------------------------------
// last arrival of a q/k group rolls the group's q/k conv_state
// ---------------------------------------------------------------------------
template <typename Act, int K, int NT>
__device__ __forceinline__ void roll_qk(const Params& p, const Item& it, int tid) {
  using AT = ActT<Act>;
  using Raw = typename AT::Raw;
  constexpr int VEC = AT::VEC;
  constexpr int NQ = K / VEC;
  const int T = p.T;
  const int dim = p.dim;
  const Act* xq = static_cast<const Act*>(p.mixed_qkv) + (size_t)it.n * T * dim;
  Act* cs_base = static_cast<Act*>(p.conv_state) + (size_t)it.n * dim * (kConvW - 1);
  for (int task = tid; task < 2 * NQ; task += NT) {
    const int c = task < NQ ? it.h * K + task * VEC : p.H * K + it.h * K + (task - NQ) * VEC;
    Act* csp = cs_base + (size_t)c * (kConvW - 1);
    Raw old[3 * VEC] = {};
    if (T < kConvW - 1) {
#pragma unroll
      for (int m = 0; m < 3; ++m)
        AT::unpack(ld_rw_16(reinterpret_cast<const char*>(csp) + 16 * m), old + m * VEC);
    }
    Raw r[3 * VEC];
#pragma unroll
    for (int j = 0; j < kConvW - 1; ++j) {
      const int idx = T + j;  // position in [state || tokens]
      Raw xv[VEC];
      if (idx >= kConvW - 1) {
        AT::unpack(ld_ro_16(xq + (size_t)(idx - (kConvW - 1)) * dim + c), xv);
#pragma unroll
        for (int e = 0; e < VEC; ++e) r[e * (kConvW - 1) + j] = xv[e];
      } else {
        // select old[.., idx] with compile-time indices only (no local memory)
#pragma unroll
        for (int jj = 0; jj < kConvW - 1; ++jj)
          if (jj == idx) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) r[e * (kConvW - 1) + j] = old[e * (kConvW - 1) + jj];
          }
      }
    }
#pragma unroll
    for (int m = 0; m < 3; ++m) st_16(reinterpret_cast<char*>(csp) + 16 * m, AT::pack(r + m * VEC));
  }
}

// Arrival of one item on its q/k group counter (thread 0 only).  Returns true
// for the last arrival, which also resets the counter.
__device__ __forceinline__ bool arrive_qk_group(const Params& p, const Item& it) {
  const int expected = p.G * p.nvt;
  if (expected == 1) return true;
  int* cnt = p.counters + (size_t)it.n * p.H + it.h;
  __threadfence();  // this CTA's conv_state reads are done (a barrier precedes)
  const int old = atomicAdd(cnt, 1);
  if (old != expected - 1) return false;
  atomicExch(cnt, 0);
  __threadfence();
  return true;
}

// ---------------------------------------------------------------------------
// consumer: the recurrence on register-resident S
// ---------------------------------------------------------------------------
template <typename Act, int K, int BV>
__device__ __forceinline__ void consume(const Params& p, const Item& it, const float* sQ,
                                       const float* sK, const float* sA, const float* sV,
                                       const float* sB, float4 (&s)[K / 8], int warp, int lane) {
  constexpr int R = K / 8;
  const int rg = lane >> 2;
  const int cg = lane & 3;
  const int col = warp * 16 + cg * 4;  // column within the tile
  const int T = p.T;
  const int V = p.V;
  const size_t colg = (size_t)it.vt * BV + col;  // column within the state
  for (int t = 0; t < T; ++t) {
    const float* al = sA + t * K + rg * R;
    const float* kk = sK + t * K + rg * R;
    const float* qq = sQ + t * K + rg * R;
    // decay, then partial S^T k over this thread's rows
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < R; i += 4) {
      const float4 a4 = *reinterpret_cast<const float4*>(al + i);
      const float4 k4 = *reinterpret_cast<const float4*>(kk + i);
      const float av[4] = {a4.x, a4.y, a4.z, a4.w};
      const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float4& x = s[i + j];
        x.x = __fmul_rn(x.x, av[j]); x.y = __fmul_rn(x.y, av[j]);
        x.z = __fmul_rn(x.z, av[j]); x.w = __fmul_rn(x.w, av[j]);
        acc.x = __fmaf_rn(x.x, kv[j], acc.x); acc.y = __fmaf_rn(x.y, kv[j], acc.y);
        acc.z = __fmaf_rn(x.z, kv[j], acc.z); acc.w = __fmaf_rn(x.w, kv[j], acc.w);
      }
    }
#pragma unroll
    for (int off = 4; off <= 16; off <<= 1) {
      acc.x = __fadd_rn(acc.x, __shfl_xor_sync(0xffffffffu, acc.x, off));
      acc.y = __fadd_rn(acc.y, __shfl_xor_sync(0xffffffffu, acc.y, off));
      acc.z = __fadd_rn(acc.z, __shfl_xor_sync(0xffffffffu, acc.z, off));
      acc.w = __fadd_rn(acc.w, __shfl_xor_sync(0xffffffffu, acc.w, off));
    }
    // u = beta (v - S^T k)
    const float4 v4 = *reinterpret_cast<const float4*>(sV + t * BV + col);
    const float be = sB[t];
    float4 u;
    u.x = __fmul_rn(be, __fsub_rn(v4.x, acc.x)); u.y = __fmul_rn(be, __fsub_rn(v4.y, acc.y));
    u.z = __fmul_rn(be, __fsub_rn(v4.z, acc.z)); u.w = __fmul_rn(be, __fsub_rn(v4.w, acc.w));
    // rank-1 update, partial S^T q, streaming snapshot store
    float* dst = p.inter_ssm + ((((size_t)it.n * T + t) * p.HV + it.hv) * K + rg * R) * V + colg;
    float4 oa = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < R; i += 4) {
      const float4 k4 = *reinterpret_cast<const float4*>(kk + i);
      const float4 q4 = *reinterpret_cast<const float4*>(qq + i);
      const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
      const float qv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float4& x = s[i + j];
        x.x = __fmaf_rn(kv[j], u.x, x.x); x.y = __fmaf_rn(kv[j], u.y, x.y);
        x.z = __fmaf_rn(kv[j], u.z, x.z); x.w = __fmaf_rn(kv[j], u.w, x.w);
        oa.x = __fmaf_rn(x.x, qv[j], oa.x); oa.y = __fmaf_rn(x.y, qv[j], oa.y);
        oa.z = __fmaf_rn(x.z, qv[j], oa.z); oa.w = __fmaf_rn(x.w, qv[j], oa.w);
        st_stream_f4(dst + (size_t)(i + j) * V, x);
      }
    }
#pragma unroll
    for (int off = 4; off <= 16; off <<= 1) {
      oa.x = __fadd_rn(oa.x, __shfl_xor_sync(0xffffffffu, oa.x, off));
      oa.y = __fadd_rn(oa.y, __shfl_xor_sync(0xffffffffu, oa.y, off));
      oa.z = __fadd_rn(oa.z, __shfl_xor_sync(0xffffffffu, oa.z, off));
      oa.w = __fadd_rn(oa.w, __shfl_xor_sync(0xffffffffu, oa.w, off));
    }
    if (rg == 0) {
      Act* op = static_cast<Act*>(p.o) + (((size_t)it.n * T + t) * p.HV + it.hv) * V + colg;
      ActT<Act>::store4(op, oa);
    }
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <typename Act, int K, int WARPS, bool PERSIST>
__global__ void __launch_bounds__(WARPS * 32, 16 / WARPS)
    kda_verify_kernel(const __grid_constant__ CUtensorMap tmap_s0, const Params p) {
  constexpr int BV = WARPS * 16;
  constexpr int NT = WARPS * 32;
  constexpr int R = K / 8;
  static_assert(K % 32 == 0 && K <= 128, "K must be 32, 64 or 128");

  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem);
  int* sflag = reinterpret_cast<int*>(smem + 8);  // [NSTAGE] last-arrival flags
  float* sbuf = reinterpret_cast<float*>(smem + 128);
  float* stage0 = sbuf + K * BV;
  const int T = p.T;
  const int sf = stage_floats(T, K, BV);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  long long item = blockIdx.x;
  if (item >= p.num_items) return;
  const long long stride = PERSIST ? (long long)gridDim.x : p.num_items;

  if (tid == 0) {
    mbar_init(mbar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const uint64_t pol = l2_policy_evict_first();
  if (tid == 0) {
    prefetch_tensormap(&tmap_s0);
    const Item it = decode_item(p, item);
    mbar_arrive_expect_tx(mbar, K * BV * sizeof(float));
    tma_load_2d(sbuf, &tmap_s0, it.vt * BV, static_cast<int>(it.unit * K), mbar, pol);
  }

  auto produce = [&](long long itm, int buf) {
    const Item it = decode_item(p, itm);
    float* st = stage0 + buf * sf;
    float* sQ = st;
    float* sK = sQ + T * K;
    float* sA = sK + T * K;
    float* sV = sA + T * K;
    float* sB = sV + T * BV;
    produce_phase1<Act, K, BV, NT>(p, it, sQ, sK, sA, sV, sB, tid);
    __syncthreads();
    if (tid == 0) sflag[buf] = arrive_qk_group(p, it) ? 1 : 0;
    produce_phase2<K, WARPS>(T, sQ, sK, warp, lane);
    __syncthreads();
  };

  produce(item, 0);
  for (int iter = 0;; ++iter) {
    const int buf = PERSIST ? (iter & 1) : 0;
    const Item it = decode_item(p, item);
    const bool ok = mbar_wait_bounded(mbar, static_cast<uint32_t>(iter & 1), kWaitLimitNs);
    if (__syncthreads_or(!ok)) {
      // give up without hanging: report, let the copy in flight land, leave
      if (tid == 0) atomicOr(p.status, 1);
      mbar_wait_bounded(mbar, static_cast<uint32_t>(iter & 1), kWaitLimitNs);
      __syncthreads();
      return;
    }
    float4 s[R];
    {
      const int rg = lane >> 2, cg = lane & 3;
      const float* src = sbuf + (rg * R) * BV + warp * 16 + cg * 4;
#pragma unroll
      for (int i = 0; i < R; ++i) s[i] = *reinterpret_cast<const float4*>(src + i * BV);
    }
    const long long next = item + stride;
    const bool has_next = PERSIST && next < p.num_items;
    if (PERSIST) {
      __syncthreads();  // every thread has copied the tile out of sbuf
      if (has_next && tid == 0) {
        fence_proxy_async_smem();
        const Item nx = decode_item(p, next);
        mbar_arrive_expect_tx(mbar, K * BV * sizeof(float));
        tma_load_2d(sbuf, &tmap_s0, nx.vt * BV, static_cast<int>(nx.unit * K), mbar, pol);
      }
    }
    {
      const float* st = stage0 + buf * sf;
      consume<Act, K, BV>(p, it, st, st + T * K, st + 2 * T * K, st + 3 * T * K,
                          st + 3 * T * K + T * BV, s, warp, lane);
    }
    if (sflag[buf]) roll_qk<Act, K, NT>(p, it, tid);
    if (!has_next) break;
    item = next;
    produce(item, buf ^ 1);
  }
}

}  // namespace kda
