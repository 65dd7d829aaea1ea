// kda_api.cu -- the C ABI declared in include/kda_verify.h: argument
// validation, the dispatcher, the TMA descriptor of the
// state tensor, and the launch.  Host code only; kernels live in
// kda_kernel.cuh and are instantiated in kda_inst_*.cu.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "kda_launch.cuh"
#include "../../include/kda_verify.h"

namespace {

using kda::LaunchCfg;
using kda::Params;

constexpr int kSmemPerSm = 233472;  // bytes of shared memory per SM (228 KB)
constexpr int kSmemReservedPerCta = 1024;
constexpr size_t kMaxSmemPerCta = 232448;  // opt-in dynamic shared memory per CTA (227 KB)

bool supported_dim(int x) { return x == 32 || x == 64 || x == 128 || x == 256; }

int check_shape(const kda_shape* s) {
  if (!s) return KDA_ERR_NULL;
  if (s->act != KDA_F32 && s->act != KDA_BF16) return KDA_ERR_DTYPE;
  if (s->N < 0 || s->T < 1 || s->T > KDA_MAX_T) return KDA_ERR_SHAPE;
  if (s->H < 1 || s->HV < s->H || s->HV % s->H != 0) return KDA_ERR_SHAPE;
  if (s->W != 4) return KDA_ERR_SHAPE;
  if (!supported_dim(s->K) || !supported_dim(s->V)) return KDA_ERR_SHAPE;
  // TMA row coordinate (N*HV*K) and element counts must fit the index types
  const long long rows = (long long)s->N * s->HV * s->K;
  if (rows >= (1ll << 31)) return KDA_ERR_SHAPE;
  return KDA_OK;
}

size_t act_bytes(const kda_shape* s) { return s->act == KDA_F32 ? 4 : 2; }

int ctas_per_sm_for(int regs_limit, size_t smem) {
  const int by_smem = (int)(kSmemPerSm / (smem + kSmemReservedPerCta));
  return std::max(1, std::min(regs_limit, by_smem));
}

// Launches of at least this many waves of resident CTAs roll the shared q/k
// conv_state with the second kernel instead of the cluster (or the counter).
constexpr int kQkRollKernelWaves = 2;

// v-tile widths of the one-item kernels: 1, 2, 4 or 8 warps of warp_cols(K)
// columns each (16 columns for K <= 128, 8 for K = 256); the shared-memory
// state variant runs 4 or 8 warps.
bool fits_v(int bv, int V) { return bv <= V && V % bv == 0; }
bool valid_tile_bv(int bv, int K, int V) {
  const int wc = kda::warp_cols(K);
  return (bv == 2 * wc || bv == 4 * wc || bv == 8 * wc || (K <= 128 && bv == wc)) && fits_v(bv, V);
}
bool valid_pipe_bv(int bv, int K, int V) {
  return K <= 128 && (bv == 4 * kda::warp_cols(K) || bv == 8 * kda::warp_cols(K)) && fits_v(bv, V);
}
bool valid_split_bv(int bv, int K, int V) {
  return K <= 128 && (bv == 2 * kda::warp_cols(K) || bv == 4 * kda::warp_cols(K) || bv == 8 * kda::warp_cols(K)) &&
         fits_v(bv, V);
}
bool valid_sms_bv(int bv, int K, int V) {
  const int wc = kda::warp_cols(K);
  return (bv == 4 * wc || bv == 8 * wc) && fits_v(bv, V);
}

// The cluster q/k roll is built for the one-item kernel with the state in
// registers at 4 or 8 warps, and for groups of at most KDA_MAX_QK_CLUSTER
// items (a portable cluster size).
bool cluster_roll_built(const kda_plan* plan, const kda_shape* s) {
  const int wc = kda::warp_cols(s->K);
  if (plan->variant != KDA_VARIANT_ONE_ITEM || (plan->bv != 4 * wc && plan->bv != 8 * wc)) return false;
  if (!valid_tile_bv(plan->bv, s->K, s->V)) return false;
  return (long long)(s->HV / s->H) * (s->V / plan->bv) <= KDA_MAX_QK_CLUSTER;
}

// A plan's tile width against its variant (decode: no pipelined variant;
// the pipelined variant is built for K <= 128 and needs its shared memory --
// two raw-input buffers and two stages besides the tile -- to fit one CTA).
bool valid_plan(const kda_plan* plan, const kda_shape* s, bool decode) {
  if (plan->qk_roll < KDA_QK_ROLL_AUTO || plan->qk_roll > KDA_QK_ROLL_CLUSTER) return false;
  const int K = s->K, V = s->V;
  if (plan->qk_roll == KDA_QK_ROLL_CLUSTER && !cluster_roll_built(plan, s)) return false;
  switch (plan->variant) {
    case KDA_VARIANT_ONE_ITEM: return valid_tile_bv(plan->bv, K, V);
    case KDA_VARIANT_PIPELINED:
      return !decode && valid_pipe_bv(plan->bv, K, V) &&
             kda::pipe_smem_bytes(s->T, K, plan->bv, (int)act_bytes(s)) <= kMaxSmemPerCta;
    case KDA_VARIANT_ONE_ITEM_SMEM: return valid_sms_bv(plan->bv, K, V);
    case KDA_VARIANT_SPLIT:
      // each item's stage must fit its home (the first rows of its K x bv slice
      // of the last token's snapshot); the prep kernel's staging one CTA
      return !decode && valid_split_bv(plan->bv, K, V) &&
             (size_t)kda::stage_floats(s->T, K, plan->bv) <= (size_t)K * plan->bv &&
             kda::prep_smem_bytes(s->T, K, V, s->HV / s->H, (int)act_bytes(s)) <= kMaxSmemPerCta;
    default: return false;
  }
}

// Fill the derived fields of a plan whose variant and bv are set.
void finish_plan(const kda_shape* s, int num_sms, kda_plan* out, int requested_grid,
                 int requested_prefetch, int requested_qk_roll) {
  const long long units = (long long)s->N * s->HV;
  const int ab = s->act == KDA_F32 ? 4 : 2;
  out->items = units * (s->V / out->bv);
  if (out->variant == KDA_VARIANT_PIPELINED) {
    out->warps = out->bv / kda::warp_cols(s->K);
    const size_t smem = kda::pipe_smem_bytes(s->T, s->K, out->bv, ab);
    out->ctas_per_sm = ctas_per_sm_for(kda::pipe_min_blocks(out->warps), smem);
    const long long cap = (long long)num_sms * out->ctas_per_sm;
    long long grid = requested_grid > 0 ? requested_grid : cap;
    out->grid = (int)std::max(1LL, std::min(out->items, grid));
    // the kernel requests every input one item ahead itself: no L2 prefetch
    out->prefetch = 0;
  } else {
    out->warps = out->bv / kda::warp_cols(s->K);
    const size_t smem = kda::tile_smem_bytes(s->T, s->K, out->bv, ab);
    const bool sms = out->variant == KDA_VARIANT_ONE_ITEM_SMEM;
    out->ctas_per_sm = ctas_per_sm_for(kda::tile_min_blocks(out->warps, sms), smem);
    // (the split variant's recurrence kernel has the one-item kernel's layout)
    out->grid = (int)std::max(1LL, out->items);
    // 3/8 of a wave of resident CTAs ahead: measured on GB300, any distance
    // between ~1/4 and ~5/8 of a wave is within 2 %; a full wave or more lets
    // the streaming snapshot writes evict the prefetched lines before use
    const int dist = std::max(1, num_sms * out->ctas_per_sm * 3 / 8);
    out->prefetch = requested_prefetch < 0 ? 0 : (requested_prefetch > 0 ? requested_prefetch : dist);
  }
  // q/k conv_state roll when several items share a group's q/k channels: the
  // counter protocol costs the verify kernel a fence and an atomic round trip
  // per item (measured on GB300: 6-14 % on launches of many waves), the second
  // kernel a launch and a dependency wait (its loads overlap the verify's
  // last wave), the cluster launch slower CTA scheduling on many waves (up to
  // 25 % at one token) but nothing per item.  Measured on GB300 over the
  // sweep's 100 points with several items per group: below 2 waves the
  // cluster is the fastest (2-6 % ahead of the second kernel, 4-8 % of the
  // counter), from about 3 waves on the second kernel (4 % at 3.4 waves)
  const bool shared_qk = (long long)(s->HV / s->H) * (s->V / out->bv) > 1;
  if (out->variant == KDA_VARIANT_SPLIT) {
    // its first kernel rolls every channel of a group: no protocol needed
    out->qk_roll = KDA_QK_ROLL_AUTO;
    out->launches = 2;
    if (units == 0) out->grid = 0;
    return;
  }
  if (!shared_qk) {
    out->qk_roll = KDA_QK_ROLL_COUNTER;
  } else if (requested_qk_roll != KDA_QK_ROLL_AUTO) {
    out->qk_roll = requested_qk_roll;
  } else {
    out->qk_roll = out->items >= (long long)kQkRollKernelWaves * num_sms * out->ctas_per_sm
                       ? KDA_QK_ROLL_KERNEL
                       : (cluster_roll_built(out, s) ? KDA_QK_ROLL_CLUSTER : KDA_QK_ROLL_COUNTER);
  }
  out->launches = (shared_qk && out->qk_roll == KDA_QK_ROLL_KERNEL) ? 2 : 1;
  if (units == 0) out->grid = 0;
}

struct Span {
  uintptr_t lo, hi;
};

bool overlap(const Span& a, const Span& b) {
  return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int num_sms_of_current_device(int* out) {
  static int cache[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  if (dev < 64 && cache[dev] > 0) {
    *out = cache[dev];
    return 0;
  }
  int n = 0;
  e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return (int)e;
  if (dev < 64) cache[dev] = n;
  *out = n;
  return 0;
}

}  // namespace

extern "C" {

int kda_version(void) { return 0x000100; }

size_t kda_workspace_bytes(const kda_shape* s) {
  if (!s) return 0;
  const size_t counters = (size_t)std::max(0, s->N) * (size_t)std::max(0, s->H);
  const size_t bytes = (counters + 4) * sizeof(int);  // counters + status word (+pad)
  return (bytes + 255) / 256 * 256;
}

}  // extern "C"

namespace {

// The dispatcher.  `decode`: plan for kda_conv_decode (one-item kernels only).
int make_plan_impl(const kda_shape* s, int num_sms, kda_variant variant, bool decode, kda_plan* out) {
  int rc = check_shape(s);
  if (rc) return rc;
  if (!out) return KDA_ERR_NULL;
  if (num_sms < 1) return KDA_ERR_DEVICE;
  if (variant != KDA_VARIANT_AUTO && variant != KDA_VARIANT_ONE_ITEM &&
      variant != KDA_VARIANT_PIPELINED && variant != KDA_VARIANT_ONE_ITEM_SMEM &&
      variant != KDA_VARIANT_SPLIT)
    return KDA_ERR_VARIANT;
  if (decode && (variant == KDA_VARIANT_PIPELINED || variant == KDA_VARIANT_SPLIT)) return KDA_ERR_VARIANT;
  const long long units = (long long)s->N * s->HV;
  std::memset(out, 0, sizeof(*out));
  // widest one-item tile: 8 warps (128 columns for K <= 128, 64 for K = 256)
  const int full_bv = std::min(s->V, 8 * kda::warp_cols(s->K));
  if (variant == KDA_VARIANT_PIPELINED) {
    out->variant = KDA_VARIANT_PIPELINED;
    out->bv = full_bv;
    if (!valid_plan(out, s, false)) {  // K > 128, V < 64, or too much shared memory
      out->bv = 4 * kda::warp_cols(s->K);
      if (!valid_plan(out, s, false)) return KDA_ERR_VARIANT;
    }
  } else if (variant == KDA_VARIANT_SPLIT) {
    out->variant = KDA_VARIANT_SPLIT;
    out->bv = full_bv;
    if (!valid_plan(out, s, false)) return KDA_ERR_VARIANT;
  } else if (variant == KDA_VARIANT_ONE_ITEM_SMEM) {
    if (s->V < 4 * kda::warp_cols(s->K)) return KDA_ERR_VARIANT;
    out->variant = KDA_VARIANT_ONE_ITEM_SMEM;
    out->bv = full_bv;
  } else {
    // One item per CTA, the state in registers: the fastest kernel at 143 of
    // the 150 points of the configuration sweep (T in 1..8, N in 1..512, three
    // head layouts, both gates; K = V = 128) and at 140 of the same 150 points
    // for the plain decode.
    out->variant = KDA_VARIANT_ONE_ITEM;
    out->bv = full_bv;
    const int G = s->HV / s->H;
    if (s->K <= 128 && full_bv == 128) {
      // Single tokens over many units: the shared-memory state (3 CTAs per SM
      // instead of 2) from 8 units per SM -- verifies with one v-head per q/k
      // head (+3..5 %) and plain decodes (+2..5 %).  From two tokens on the
      // register-state decode kernels are faster.
      const long long smem_from = (s->T == 1 && (decode || G == 1)) ? 8 : 0;
      const bool few = !decode && 2 * units <= num_sms;
      if (smem_from > 0 && units >= smem_from * num_sms) {
        out->variant = KDA_VARIANT_ONE_ITEM_SMEM;
      } else if ((G >= 2 && s->T <= 2) || few) {
        // 64-column tiles (twice the CTAs): with several v-heads per q/k head
        // for calls of up to two tokens (+2..17 %), and for verifies of at
        // most half a unit per SM, where the idle SMs absorb the repeated
        // q/k work (+5..10 % at one token, even at other T).  Longer calls
        // keep 128 columns: each 64-column item repeats the q/k conv of all T
        // tokens (up to 20 % slower for plain decodes of three tokens).
        out->bv = 4 * kda::warp_cols(s->K);
      }
    } else if (decode && s->T == 1 && units >= 8LL * num_sms && valid_sms_bv(full_bv, s->K, s->V)) {
      // The other head dims' plain decode of one token over many units: the
      // shared-memory state too (K = V = 64: +3.5 %, K = V = 256: +4 %); their
      // verifies keep the register state (1-2 % faster there).
      out->variant = KDA_VARIANT_ONE_ITEM_SMEM;
    }
  }
  finish_plan(s, num_sms, out, 0, 0, KDA_QK_ROLL_AUTO);
  return KDA_OK;
}

}  // namespace

extern "C" {

int kda_make_plan(const kda_shape* s, int num_sms, kda_variant variant, kda_plan* out) {
  return make_plan_impl(s, num_sms, variant, false, out);
}

int kda_make_decode_plan(const kda_shape* s, int num_sms, kda_variant variant, kda_plan* out) {
  return make_plan_impl(s, num_sms, variant, true, out);
}

int kda_resolve_plan(const kda_shape* s, int num_sms, int decode, kda_plan* plan) {
  int rc = check_shape(s);
  if (rc) return rc;
  if (!plan) return KDA_ERR_NULL;
  if (num_sms < 1) return KDA_ERR_DEVICE;
  if (!valid_plan(plan, s, decode != 0)) return KDA_ERR_VARIANT;
  finish_plan(s, num_sms, plan, plan->grid, plan->prefetch, plan->qk_roll);
  return KDA_OK;
}

}  // extern "C"

namespace {

// Every host-side check of one call (nothing touches the GPU).
// Slots of the three state pools (identity and N slots for the dense calls).
struct Pools {
  const int32_t* idx_state = nullptr;
  const int32_t* idx_conv = nullptr;
  const int32_t* idx_inter = nullptr;
  size_t n_state = 0, n_conv = 0, n_inter = 0;
};

Pools dense_pools(const kda_shape* s) {
  Pools pl;
  pl.n_state = pl.n_conv = pl.n_inter = (size_t)std::max(0, s->N);
  return pl;
}

int pools_from(const kda_shape* s, const kda_state_indices* idx, Pools* out) {
  *out = dense_pools(s);
  if (!idx) return KDA_OK;
  auto one = [&](const int32_t* ix, int pool, const int32_t** dst, size_t* n) {
    if (!ix) return KDA_OK;
    if (pool < 1) return KDA_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(ix) & 3u) return KDA_ERR_MISALIGNED;
    *dst = ix;
    *n = (size_t)pool;
    return KDA_OK;
  };
  int rc = one(idx->cache_indices, idx->state_pool, &out->idx_state, &out->n_state);
  if (!rc) rc = one(idx->conv_state_indices, idx->conv_pool, &out->idx_conv, &out->n_conv);
  if (!rc) rc = one(idx->intermediate_state_indices, idx->inter_pool, &out->idx_inter, &out->n_inter);
  if (!rc && (long long)out->n_state * s->HV * s->K >= (1ll << 31)) rc = KDA_ERR_SHAPE;
  return rc;
}

int validate_call(const kda_shape* s, const void* mixed_qkv, const void* conv_w,
                  void* conv_state, const float* A_log, const float* dt_bias, const void* a,
                  const void* b, const float* S0, kda_gate_mode gate_mode, void* o,
                  float* inter_ssm, void* conv_snapshots, void* workspace,
                  size_t workspace_bytes, const Pools& pl) {
  int rc = check_shape(s);
  if (rc) return rc;
  if (gate_mode != KDA_GATE_SOFTPLUS && gate_mode != KDA_GATE_SAFE) return KDA_ERR_GATE;
  if (s->N == 0) return KDA_OK;
  if (!mixed_qkv || !conv_w || !conv_state || !a || !b || !S0 || !o || !inter_ssm ||
      !conv_snapshots)
    return KDA_ERR_NULL;
  if (gate_mode == KDA_GATE_SOFTPLUS && (!A_log || !dt_bias)) return KDA_ERR_GATE;
  if (!workspace || workspace_bytes < kda_workspace_bytes(s)) return KDA_ERR_WORKSPACE;

  const size_t ab = act_bytes(s);
  const size_t N = s->N, T = s->T, H = s->H, HV = s->HV, K = s->K, V = s->V;
  const size_t dim = 2 * H * K + HV * V;
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!al16(mixed_qkv) || !al16(conv_w) || !al16(conv_state) || !al16(a) || !al16(S0) ||
      !al16(o) || !al16(inter_ssm) || !al16(conv_snapshots) || !al16(workspace) ||
      (reinterpret_cast<uintptr_t>(b) % ab) != 0)
    return KDA_ERR_MISALIGNED;
  if (gate_mode == KDA_GATE_SOFTPLUS && (!al16(A_log) || !al16(dt_bias)))
    return KDA_ERR_MISALIGNED;

  auto span = [](const void* p, size_t bytes) {
    Span sp;
    sp.lo = reinterpret_cast<uintptr_t>(p);
    sp.hi = sp.lo + (p ? bytes : 0);
    return sp;
  };
  const Span in[] = {
      span(mixed_qkv, N * T * dim * ab), span(conv_w, dim * 4 * ab),
      span(gate_mode == KDA_GATE_SOFTPLUS ? A_log : nullptr, HV * 4),
      span(gate_mode == KDA_GATE_SOFTPLUS ? dt_bias : nullptr, HV * K * 4),
      span(a, N * T * HV * K * ab), span(b, N * T * HV * ab),
      span(S0, pl.n_state * HV * K * V * 4), span(pl.idx_state, N * 4), span(pl.idx_conv, N * 4),
      span(pl.idx_inter, N * 4)};
  const Span wr[] = {span(conv_state, pl.n_conv * dim * 3 * ab), span(o, N * T * HV * V * ab),
                     span(inter_ssm, pl.n_inter * T * HV * K * V * 4),
                     span(conv_snapshots, pl.n_inter * T * dim * 3 * ab),
                     span(workspace, kda_workspace_bytes(s))};
  for (size_t i = 0; i < sizeof(wr) / sizeof(wr[0]); ++i) {
    for (const Span& x : in)
      if (overlap(wr[i], x)) return KDA_ERR_ALIAS;
    for (size_t j = 0; j < sizeof(wr) / sizeof(wr[0]); ++j)
      if (j != i && overlap(wr[i], wr[j])) return KDA_ERR_ALIAS;
  }
  return KDA_OK;
}

// Encode the state tensor map and launch the kernel of `plan`.
int launch_plan(const kda_shape* s, const void* mixed_qkv, const void* conv_w, void* conv_state,
                const float* A_log, const float* dt_bias, const void* a, const void* b,
                const float* S0, kda_gate_mode gate_mode, void* o, float* inter_ssm,
                void* conv_snapshots, void* workspace, const kda_plan& plan, const Pools& pl,
                kda_stream_t stream, float* S_out = nullptr) {
  const size_t N = s->N, H = s->H, HV = s->HV, K = s->K, V = s->V;
  const size_t dim = 2 * H * K + HV * V;
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return KDA_ERR_DEVICE;
  CUtensorMap tmap;
  std::memset(&tmap, 0, sizeof(tmap));
  cuuint64_t gdim[2] = {(cuuint64_t)V, (cuuint64_t)(pl.n_state * HV * K)};
  cuuint64_t gstride[1] = {(cuuint64_t)(V * sizeof(float))};
  // the kernels load a tile as boxes of 32 columns (128 bytes) with the
  // 128-byte swizzle, or as one row-major box when the tile is narrower
  const bool swz = plan.bv >= 32;
  cuuint32_t box[2] = {(cuuint32_t)kda::tile_box_cols(plan.bv), (cuuint32_t)K};
  cuuint32_t estride[2] = {1, 1};
  CUresult cr = encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(S0), gdim,
                       gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                       swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return KDA_ERR_DEVICE;

  Params p;
  p.mixed_qkv = mixed_qkv;
  p.conv_w = conv_w;
  p.conv_state = conv_state;
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.a = a;
  p.b = b;
  p.o = o;
  p.inter_ssm = inter_ssm;
  p.conv_snapshots = conv_snapshots;
  p.S_out = S_out;
  p.counters = static_cast<int*>(workspace);
  p.status = static_cast<int*>(workspace) + N * H;
  p.num_items = plan.items;
  p.prefetch = plan.prefetch;
  p.idx_state = pl.idx_state;
  p.idx_conv = pl.idx_conv;
  p.idx_inter = pl.idx_inter;
  p.pool_state = (int)pl.n_state;
  p.pool_conv = (int)pl.n_conv;
  p.pool_inter = (int)pl.n_inter;
  p.N = s->N;
  p.T = s->T;
  p.H = s->H;
  p.HV = s->HV;
  p.V = s->V;
  p.dim = (int)dim;
  p.G = s->HV / s->H;
  p.nvt = s->V / plan.bv;
  p.gate_mode = gate_mode == KDA_GATE_SOFTPLUS ? 0 : 1;
  p.div_nvt = kda::make_fastdiv((uint32_t)p.nvt);
  p.div_HV = kda::make_fastdiv((uint32_t)p.HV);
  p.div_G = kda::make_fastdiv((uint32_t)p.G);
  p.div_T = kda::make_fastdiv((uint32_t)p.T);
  const bool roll_kernel = plan.qk_roll == KDA_QK_ROLL_KERNEL && p.G * p.nvt > 1;
  p.qk_roll_kernel = roll_kernel ? 1 : 0;
  // (valid_plan admits the cluster roll only where it is built)
  p.qk_cluster = plan.qk_roll == KDA_QK_ROLL_CLUSTER && p.G * p.nvt > 1 ? p.G * p.nvt : 0;

  LaunchCfg cfg;
  cfg.K = s->K;
  cfg.warps = plan.warps;
  cfg.pipe = plan.variant == KDA_VARIANT_PIPELINED;
  cfg.split = plan.variant == KDA_VARIANT_SPLIT;
  if (cfg.split) p.qk_roll_kernel = 0;
  cfg.decode = S_out != nullptr;
  cfg.sms = plan.variant == KDA_VARIANT_ONE_ITEM_SMEM;
  cfg.grid = plan.grid;
  const int ab = s->act == KDA_F32 ? 4 : 2;
  cfg.smem = cfg.pipe ? kda::pipe_smem_bytes(s->T, s->K, plan.bv, ab)
                      : kda::tile_smem_bytes(s->T, s->K, plan.bv, ab);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int rc;
  if (cfg.split) {
    const size_t prep_smem = kda::prep_smem_bytes(s->T, s->K, s->V, s->HV / s->H, ab);
    rc = s->act == KDA_BF16 ? kda::launch_split_bf16(tmap, p, cfg, prep_smem, st)
                            : kda::launch_split_f32(tmap, p, cfg, prep_smem, st);
    return rc < 0 ? KDA_ERR_SHAPE : rc;
  }
  // decode launches whose q/k conv_state needs no counter run the
  // counter-free decode kernels
  const bool counter_free = cfg.decode && !cfg.pipe && (p.G * p.nvt == 1 || p.qk_roll_kernel);
  if (p.qk_cluster > 1)
    rc = s->act == KDA_BF16 ? kda::launch_tile_cluster_bf16(tmap, p, cfg, st)
                            : kda::launch_tile_cluster_f32(tmap, p, cfg, st);
  else if (counter_free)
    rc = s->act == KDA_BF16 ? kda::launch_tile_decode_bf16(tmap, p, cfg, st)
                            : kda::launch_tile_decode_f32(tmap, p, cfg, st);
  else if (s->act == KDA_BF16)
    rc = cfg.pipe ? kda::launch_pipe_bf16(tmap, p, cfg, st) : kda::launch_tile_bf16(tmap, p, cfg, st);
  else
    rc = cfg.pipe ? kda::launch_pipe_f32(tmap, p, cfg, st) : kda::launch_tile_f32(tmap, p, cfg, st);
  if (rc < 0) return KDA_ERR_SHAPE;
  if (rc == 0 && roll_kernel) rc = kda::launch_qk_roll(p, s->K, s->act == KDA_BF16, st);
  return rc;
}

}  // namespace

extern "C" {

int kda_conv_verify_variant(const kda_shape* s, const void* mixed_qkv, const void* conv_w,
                            void* conv_state, const float* A_log, const float* dt_bias,
                            const void* a, const void* b, const float* S0,
                            kda_gate_mode gate_mode, void* o, float* inter_ssm,
                            void* conv_snapshots, void* workspace, size_t workspace_bytes,
                            kda_variant variant, kda_stream_t stream) {
  if (variant != KDA_VARIANT_AUTO && variant != KDA_VARIANT_ONE_ITEM &&
      variant != KDA_VARIANT_PIPELINED && variant != KDA_VARIANT_ONE_ITEM_SMEM &&
      variant != KDA_VARIANT_SPLIT)
    return KDA_ERR_VARIANT;
  if (!s) return KDA_ERR_NULL;
  const Pools pl = dense_pools(s);
  int rc = validate_call(s, mixed_qkv, conv_w, conv_state, A_log, dt_bias, a, b, S0, gate_mode,
                         o, inter_ssm, conv_snapshots, workspace, workspace_bytes, pl);
  if (rc || s->N == 0) return rc;
  int num_sms = 0;
  rc = num_sms_of_current_device(&num_sms);
  if (rc) return rc;
  kda_plan plan;
  rc = kda_make_plan(s, num_sms, variant, &plan);
  if (rc) return rc;
  return launch_plan(s, mixed_qkv, conv_w, conv_state, A_log, dt_bias, a, b, S0, gate_mode, o,
                     inter_ssm, conv_snapshots, workspace, plan, pl, stream);
}

}  // extern "C"

namespace {

// Shared tail of the explicit-plan and indexed entry points.
int verify_with(const kda_shape* s, const Pools& pl, const void* mixed_qkv, const void* conv_w,
                void* conv_state, const float* A_log, const float* dt_bias, const void* a,
                const void* b, const float* S0, kda_gate_mode gate_mode, void* o, float* inter_ssm,
                void* conv_snapshots, void* workspace, size_t workspace_bytes, const kda_plan* plan,
                kda_stream_t stream) {
  int rc = validate_call(s, mixed_qkv, conv_w, conv_state, A_log, dt_bias, a, b, S0, gate_mode,
                         o, inter_ssm, conv_snapshots, workspace, workspace_bytes, pl);
  if (rc || s->N == 0) return rc;
  if (plan && !valid_plan(plan, s, false)) return KDA_ERR_VARIANT;
  int num_sms = 0;
  rc = num_sms_of_current_device(&num_sms);
  if (rc) return rc;
  kda_plan p;
  if (!plan) {
    rc = kda_make_plan(s, num_sms, KDA_VARIANT_AUTO, &p);
    if (rc) return rc;
  } else {
    p = *plan;
    finish_plan(s, num_sms, &p, plan->grid, plan->prefetch, plan->qk_roll);
  }
  return launch_plan(s, mixed_qkv, conv_w, conv_state, A_log, dt_bias, a, b, S0, gate_mode, o,
                     inter_ssm, conv_snapshots, workspace, p, pl, stream);
}

}  // namespace

extern "C" {

int kda_conv_verify_plan(const kda_shape* s, const void* mixed_qkv, const void* conv_w,
                         void* conv_state, const float* A_log, const float* dt_bias,
                         const void* a, const void* b, const float* S0, kda_gate_mode gate_mode,
                         void* o, float* inter_ssm, void* conv_snapshots, void* workspace,
                         size_t workspace_bytes, const kda_plan* plan, kda_stream_t stream) {
  if (!plan || !s) return KDA_ERR_NULL;
  return verify_with(s, dense_pools(s), mixed_qkv, conv_w, conv_state, A_log, dt_bias, a, b, S0,
                     gate_mode, o, inter_ssm, conv_snapshots, workspace, workspace_bytes, plan,
                     stream);
}

int kda_conv_verify_indexed(const kda_shape* s, const kda_state_indices* idx,
                            const void* mixed_qkv, const void* conv_w, void* conv_state,
                            const float* A_log, const float* dt_bias, const void* a,
                            const void* b, const float* S0, kda_gate_mode gate_mode, void* o,
                            float* inter_ssm, void* conv_snapshots, void* workspace,
                            size_t workspace_bytes, const kda_plan* plan, kda_stream_t stream) {
  if (!s) return KDA_ERR_NULL;
  int rc = check_shape(s);
  if (rc) return rc;
  Pools pl;
  rc = pools_from(s, idx, &pl);
  if (rc) return rc;
  return verify_with(s, pl, mixed_qkv, conv_w, conv_state, A_log, dt_bias, a, b, S0, gate_mode, o,
                     inter_ssm, conv_snapshots, workspace, workspace_bytes, plan, stream);
}

int kda_conv_decode(const kda_shape* s, const kda_state_indices* idx, const void* mixed_qkv,
                    const void* conv_w, void* conv_state, const float* A_log,
                    const float* dt_bias, const void* a, const void* b, float* S,
                    kda_gate_mode gate_mode, void* o, void* workspace, size_t workspace_bytes,
                    const kda_plan* plan, kda_stream_t stream) {
  if (!s) return KDA_ERR_NULL;
  int rc = check_shape(s);
  if (rc) return rc;
  if (gate_mode != KDA_GATE_SOFTPLUS && gate_mode != KDA_GATE_SAFE) return KDA_ERR_GATE;
  Pools pl;
  kda_state_indices no_inter;
  if (idx) {  // decode writes no snapshots: the intermediate slots do not apply
    no_inter = *idx;
    no_inter.intermediate_state_indices = nullptr;
  }
  rc = pools_from(s, idx ? &no_inter : nullptr, &pl);
  if (rc) return rc;
  if (s->N == 0) return KDA_OK;
  if (!mixed_qkv || !conv_w || !conv_state || !a || !b || !S || !o) return KDA_ERR_NULL;
  if (gate_mode == KDA_GATE_SOFTPLUS && (!A_log || !dt_bias)) return KDA_ERR_GATE;
  if (!workspace || workspace_bytes < kda_workspace_bytes(s)) return KDA_ERR_WORKSPACE;
  const size_t ab = act_bytes(s);
  const size_t N = s->N, T = s->T, H = s->H, HV = s->HV, K = s->K, V = s->V;
  const size_t dim = 2 * H * K + HV * V;
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!al16(mixed_qkv) || !al16(conv_w) || !al16(conv_state) || !al16(a) || !al16(S) ||
      !al16(o) || !al16(workspace) || (reinterpret_cast<uintptr_t>(b) % ab) != 0)
    return KDA_ERR_MISALIGNED;
  if (gate_mode == KDA_GATE_SOFTPLUS && (!al16(A_log) || !al16(dt_bias))) return KDA_ERR_MISALIGNED;
  auto span = [](const void* p, size_t bytes) {
    Span sp;
    sp.lo = reinterpret_cast<uintptr_t>(p);
    sp.hi = sp.lo + (p ? bytes : 0);
    return sp;
  };
  const Span in[] = {span(mixed_qkv, N * T * dim * ab), span(conv_w, dim * 4 * ab),
                     span(gate_mode == KDA_GATE_SOFTPLUS ? A_log : nullptr, HV * 4),
                     span(gate_mode == KDA_GATE_SOFTPLUS ? dt_bias : nullptr, HV * K * 4),
                     span(a, N * T * HV * K * ab), span(b, N * T * HV * ab),
                     span(pl.idx_state, N * 4), span(pl.idx_conv, N * 4)};
  const Span wr[] = {span(conv_state, pl.n_conv * dim * 3 * ab), span(S, pl.n_state * HV * K * V * 4),
                     span(o, N * T * HV * V * ab), span(workspace, kda_workspace_bytes(s))};
  for (size_t i = 0; i < sizeof(wr) / sizeof(wr[0]); ++i) {
    for (const Span& x : in)
      if (overlap(wr[i], x)) return KDA_ERR_ALIAS;
    for (size_t j = 0; j < sizeof(wr) / sizeof(wr[0]); ++j)
      if (j != i && overlap(wr[i], wr[j])) return KDA_ERR_ALIAS;
  }
  // decode runs the one-item-per-CTA kernels only
  if (plan && !valid_plan(plan, s, true)) return KDA_ERR_VARIANT;
  int num_sms = 0;
  rc = num_sms_of_current_device(&num_sms);
  if (rc) return rc;
  kda_plan p;
  if (plan) {
    p = *plan;
    finish_plan(s, num_sms, &p, plan->grid, plan->prefetch, plan->qk_roll);
  } else {
    rc = make_plan_impl(s, num_sms, KDA_VARIANT_AUTO, true, &p);
    if (rc) return rc;
  }
  return launch_plan(s, mixed_qkv, conv_w, conv_state, A_log, dt_bias, a, b, S, gate_mode, o,
                     nullptr, nullptr, workspace, p, pl, stream, S);
}

int kda_conv_verify(const kda_shape* s, const void* mixed_qkv, const void* conv_w,
                    void* conv_state, const float* A_log, const float* dt_bias, const void* a,
                    const void* b, const float* S0, kda_gate_mode gate_mode, void* o,
                    float* inter_ssm, void* conv_snapshots, void* workspace,
                    size_t workspace_bytes, kda_stream_t stream) {
  return kda_conv_verify_variant(s, mixed_qkv, conv_w, conv_state, A_log, dt_bias, a, b, S0,
                                 gate_mode, o, inter_ssm, conv_snapshots, workspace,
                                 workspace_bytes, KDA_VARIANT_AUTO, stream);
}

int kda_read_status(const kda_shape* s, void* workspace, int* status, kda_stream_t stream) {
  int rc = check_shape(s);
  if (rc) return rc;
  if (!workspace || !status) return KDA_ERR_NULL;
  int* dev_status = static_cast<int*>(workspace) + (size_t)s->N * s->H;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(status, dev_status, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && *status != 0) e = cudaMemsetAsync(dev_status, 0, sizeof(int), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return (int)e;
}

const char* kda_strerror(int code) {
  switch (code) {
    case KDA_OK: return "success";
    case KDA_ERR_NULL: return "a required pointer is NULL";
    case KDA_ERR_SHAPE: return "unsupported or inconsistent shape";
    case KDA_ERR_DTYPE: return "unknown activation dtype";
    case KDA_ERR_MISALIGNED: return "a pointer is not 16-byte aligned";
    case KDA_ERR_ALIAS: return "an output buffer overlaps an input or another output";
    case KDA_ERR_WORKSPACE: return "workspace missing or too small";
    case KDA_ERR_GATE: return "unknown gate mode, or softplus gate without A_log/dt_bias";
    case KDA_ERR_VARIANT: return "unknown kernel variant";
    case KDA_ERR_DEVICE: return "device query or driver entry point failed";
    case KDA_ERR_SCRATCH_LIMIT:
      return "shape needs more scratch than the no-alloc entry point's built-in array holds";
    default: break;
  }
  if (code > 0) return cudaGetErrorString(static_cast<cudaError_t>(code));
  return "unknown error";
}

}  // extern "C"
