// kda_kernel.cuh -- the fused causal-conv1d + KDA verify-decode kernels for
// sm_103a ("[KDA] Fuse causal conv1d into MTP verify decode", cuLA pull
// request 107).
//
// Work item: (sequence n, value head hv, v-tile vt) = a K x BV slice of one
// recurrent state, BV = warp_cols(K) * (consumer warps).
//
//   producer  conv1d(W=4) + SiLU of the q/k channels of head h = hv / G and of
//             the tile's v channels, one task per (8-channel vector, token);
//             q/k L2 norm (q scaled by K^-1/2), alpha = exp(g) and beta,
//             staged in shared memory; the raw conv windows are streamed out
//             as snapshots and the conv_state is rolled.
//   state     the item's S0 slice arrives in shared memory by 2-D TMA tile
//             loads (mbarrier completion), then moves to registers (or stays
//             in shared memory in the SMS variant).
//   consumer  a warp is RG row groups x 32/RG column quads (RG = 8 for
//             K <= 128: 16 columns per warp; RG = 16 for K = 256: 8 columns);
//             lane (rg, cg) keeps rows RG i + row_perm(rg), i < K/RG, x 4
//             columns of S.  Per token: decay + S^T k partial sums, an xor
//             butterfly across the row groups, the rank-1 update fused with
//             the S^T q partial sums and the 16-byte streaming store of the
//             snapshot, a second butterfly, o.
//
// Kernels that run that same producer arithmetic and consumer code:
//   kda_tile_kernel  one item per CTA; every warp produces, then consumes.
//                    Thread 0 issues the state-tile TMA load while its own
//                    first producer loads are in flight.  The hardware block
//                    scheduler keeps several CTAs in different phases on
//                    every SM.  Instantiated with the state in registers or
//                    in shared memory (SMS), as the plain decode (DEC: no
//                    snapshots, the final state written in place) and as the
//                    split variant's recurrence (PRE: the stage comes from
//                    kda_prep_kernel).
//   kda_pipe_kernel  persistent and warp-specialised: producer warps stage
//                    the NEXT item -- its raw inputs arrive by 1-D bulk TMA
//                    copies, its state tile by a 2-D TMA load as soon as the
//                    consumers have moved the current tile to registers --
//                    while the consumer warps stream the recurrence of the
//                    current item.  Full/empty mbarriers hand stages and tiles
//                    over; every wait is bounded.
//   kda_prep_kernel  the split variant's first kernel: the producer work of
//                    one q/k group, once, for all the items that read it.
// Same floating-point operations in the same order => bit-identical outputs.
//
// Shared q/k conv_state write-back: the q/k channels of group (n, h) are read
// by G * (V / BV) items.  With one reader it rolls them itself.  Otherwise
// a separate kernel launched after this one rolls them (kda_roll.cu;
// Params::qk_roll_kernel), or the items of the group run as one thread-block
// cluster whose first CTA rolls after the cluster barrier (the one-item
// kernel's kRollCluster instantiations), or each item arrives on a per-group
// counter after its reads and the last arrival rolls the group's q/k
// conv_state and resets the counter to zero (in the split variant the prep
// kernel rolls every channel of its group).  No CTA spins on another; the
// cluster barrier is a hardware barrier every CTA of the cluster reaches
// before any wait of its own.  v channels
// belong to exactly one item, which rolls them itself.  In the one-item
// kernel, whose threads read conv_state straight from global memory, the
// producer stages the new windows in shared memory and every roll is stored
// after the barrier that ends the CTA's conv_state reads; the pipelined kernel
// reads its raw inputs from shared memory and rolls directly.
//
// Launch overlap: every kernel here is launched as a programmatic dependent
// of whatever kernel precedes it on the stream.  Its first global access
// comes after a wait for that kernel (griddepcontrol.wait: completed, writes
// visible), and it triggers its own dependents only after that wait, so its
// launch and CTA start overlap the previous kernel's last wave while no
// access of its own, nor of a dependent that loads ahead of its own wait (the
// q/k roll kernel, the split variant's recurrence kernel), can run before the
// previous kernel's writes.  The split recurrence kernel waits for its prep
// kernel instead, which has waited for the kernel before it.
#pragma once

#include "kda_device.cuh"
#include <type_traits>

namespace kda {

// Division of numerators below 2^31 by a divisor d that is fixed for the
// whole launch (1 <= d < 2^31), by one widening multiply and a shift: the
// method of Granlund and Montgomery ("Division by invariant integers using
// multiplication", PLDI 1994).  With l = ceil(log2 d) and
// m = floor(2^(31 + l) / d) + 1, m d = 2^(31 + l) + e with 0 < e <= d <= 2^l;
// for x = q d + r (0 <= r < d, x < 2^31), m x / 2^(31 + l) = q + (r + e x /
// 2^(31 + l)) / d, and e x / 2^(31 + l) < 1, so the fraction stays below 1 and
// floor(m x / 2^(31 + l)) = q exactly; m < 2^32 because d > 2^(l - 1).  The
// item decode divides three times in a row before any load can be addressed,
// and the hardware sequence of one 32-bit division is a chain of ~20
// dependent instructions.
struct FastDiv {
  uint32_t m;  // multiplier
  uint32_t s;  // 31 + l
};

inline FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  FastDiv f;
  f.m = static_cast<uint32_t>((1ull << (31 + l)) / d + 1);
  f.s = 31 + l;
  return f;
}

__host__ __device__ __forceinline__ uint32_t fdiv(uint32_t x, FastDiv f) {
  return static_cast<uint32_t>((static_cast<uint64_t>(x) * f.m) >> f.s);
}

struct Params {
  const void* mixed_qkv;  // act [N, T, dim]
  const void* conv_w;     // act [dim, 4]
  void* conv_state;       // act [N, dim, 3]
  const float* A_log;     // f32 [HV]
  const float* dt_bias;   // f32 [HV, K]
  const void* a;          // act [N, T, HV, K]
  const void* b;          // act [N, T, HV]
  void* o;                // act [N, T, HV, V]
  float* inter_ssm;       // f32 [N, T, HV, K, V] (unused by the decode kernels)
  void* conv_snapshots;   // act [N, T, dim, 3]   (unused by the decode kernels)
  float* S_out;           // decode kernels: the final state, written in place over S0
  int* counters;          // [N * H]
  int* status;            // device status word
  long long num_items;    // N * HV * nvt
  long long prefetch;     // one-item-per-CTA kernel: L2-prefetch item + prefetch (0: off)
  // optional state-pool slots per sequence (NULL: slot = n); a negative slot
  // marks a padding sequence, which is skipped entirely
  const int* idx_state;   // S0 slot        (pool of pool_state states)
  const int* idx_conv;    // conv_state slot (pool of pool_conv windows)
  const int* idx_inter;   // inter_ssm / conv_snapshots slot (pool of pool_inter)
  int pool_state, pool_conv, pool_inter;
  int N, T, H, HV, V, dim, G, nvt;
  int gate_mode;          // 0 softplus, 1 safe
  // one-item kernels with G * nvt > 1: 1 = the q/k conv_state is rolled by
  // the separate roll kernel (no arrival counters), 0 = by the last arrival
  // or, with qk_cluster set, by the cluster
  int qk_roll_kernel;
  FastDiv div_nvt, div_HV, div_G, div_T;  // the divisors of the item and task decodes
  // one-item kernels: > 1 = the launch is made of clusters of this many CTAs,
  // the G * nvt items of one q/k group (the kernel's kRollCluster instantiation)
  int qk_cluster;
};

constexpr int kConvW = 4;
constexpr float kL2Eps = 1e-6f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kStatusTmaTimeout = 1;              // KDA_STATUS_TMA_TIMEOUT
constexpr int kStatusBadIndex = 4;                // KDA_STATUS_BAD_INDEX

__host__ __device__ constexpr int round4(int x) { return (x + 3) & ~3; }
__host__ __device__ constexpr size_t round16(size_t x) { return (x + 15) & ~size_t(15); }

// Consumer layout: a warp is RG row groups x CQ = 32 / RG column quads.
// K <= 128 uses RG = 8 (16 columns per warp, K/8 rows per thread); K = 256
// uses RG = 16 (8 columns per warp, 16 rows per thread), so a thread never
// holds more than 16 x 4 fp32 state values (64 registers).
__host__ __device__ constexpr int row_groups(int K) { return K > 128 ? 16 : 8; }
__host__ __device__ constexpr int warp_cols(int K) { return 4 * (32 / row_groups(K)); }
__host__ __device__ constexpr int rows_per_thread(int K) { return K / row_groups(K); }

// A staged K-vector (q, k or alpha of one token) is held as RG row-group
// blocks of K/RG values (see stage_pos).  Blocks are stage_rs(K) floats apart:
// K/RG rounded so that stride/4 is odd, which spreads the blocks evenly over
// the eight 16-byte bank groups, so the consumers' 16-byte reads of them (one
// block per row group) take the fewest shared-memory wavefronts.
__host__ __device__ constexpr int stage_rs(int K) {
  return rows_per_thread(K) + (((rows_per_thread(K) / 4) & 1) ? 0 : 4);
}
__host__ __device__ constexpr int stage_ks(int K) { return row_groups(K) * stage_rs(K); }

// floats of one stage: q[T][KS], k[T][KS], alpha[T][KS], v[T][BV],
// beta[round4(T)] with KS = stage_ks(K)
__host__ __device__ constexpr int stage_floats(int T, int K, int BV) {
  return 3 * T * stage_ks(K) + T * BV + round4(T);
}

// bytes of the one-item kernel's staged conv windows: x_ext[T .. T+2] of every
// channel of the item (2K + BV channels x 3 values), written by the producer
// and stored to conv_state once no reader of it is left
__host__ __device__ constexpr size_t roll_stash_bytes(int K, int BV, int ab) {
  return (size_t)(2 * K + BV) * 3 * ab;
}

// dynamic shared memory of the two kernels: 128 header bytes (mbarriers,
// flags), up to 1023 bytes of padding so that the state tile starts on a
// 1024-byte boundary (the 128-byte swizzle pattern repeats every 1024 bytes),
// the tile, then the stage(s)
constexpr size_t kSmemHeader = 128 + 1024;
__host__ __device__ constexpr size_t tile_smem_bytes(int T, int K, int BV, int ab) {
  return kSmemHeader + sizeof(float) * ((size_t)K * BV + stage_floats(T, K, BV)) +
         roll_stash_bytes(K, BV, ab);
}

// ---------------------------------------------------------------------------
// state-tile layout and row ownership
// ---------------------------------------------------------------------------
// Consumer thread (row group rg, column quad cg) owns rows RG i + row_perm(rg),
// i < K/RG.  RG = 8: row_perm = 0 4 1 5 2 6 3 7, so the two row groups that
// share a shared-memory phase (8 lanes) read rows four apart, which the
// 128-byte swizzle places in opposite halves of the banks.  RG = 16:
// row_perm(8h + 4b + j) = 8h + 2j + b, so the four row groups of a phase read
// rows whose (row mod 8) are b, b+2, b+4, b+6, four distinct swizzle offsets
// for each of the phase's two column quads.  Either way tile reads are
// conflict-free.  q, k and alpha are staged in the matching order
// (stage_pos), so a thread's K/RG values sit next to each other.
template <int K>
__device__ __forceinline__ int row_perm(int rg) {
  if constexpr (row_groups(K) == 8) {
    return (rg >> 1) + 4 * (rg & 1);
  } else {
    return ((rg >> 2) & 1) + 2 * (rg & 3) + 8 * (rg >> 3);
  }
}
template <int K>
__device__ __forceinline__ int own_row(int rg, int i) { return row_groups(K) * i + row_perm<K>(rg); }
template <int K>
__device__ __forceinline__ int stage_pos(int k) {
  constexpr int RG = row_groups(K);
  const int m = k % RG;
  int g;  // the row group that owns row k (inverse of row_perm)
  if constexpr (RG == 8) {
    g = m < 4 ? 2 * m : 2 * (m - 4) + 1;
  } else {
    g = 8 * (m >> 3) + 4 * (m & 1) + ((m >> 1) & 3);
  }
  return g * stage_rs(K) + k / RG;
}

// The tile as TMA leaves it: for BV >= 32, 32-column boxes of K rows x 128
// bytes with the 128-byte swizzle (16-byte chunk c of row k stored at chunk
// c ^ (k & 7)); narrower tiles row-major.
__host__ __device__ constexpr int tile_box_cols(int BV) { return BV >= 32 ? 32 : BV; }
template <int K, int BV>
__device__ __forceinline__ int tile_index(int k, int col) {
  if constexpr (BV >= 32) {
    return (col >> 5) * (K * 32) + k * 32 + ((((col >> 2) & 7) ^ (k & 7)) << 2) + (col & 3);
  } else {
    return k * BV + col;
  }
}

// Start of the state tile: after the header, on a 1024-byte boundary.
__device__ __forceinline__ float* tile_base(unsigned char* smem) {
  const uint32_t a = smem_u32(smem) + 128;
  return reinterpret_cast<float*>(smem + 128 + ((1024u - (a & 1023u)) & 1023u));
}

// TMA loads of one tile (one per box), all completing on `bar`.
template <int K, int BV>
__device__ __forceinline__ void tma_load_tile(float* tile, const CUtensorMap* map, int vt,
                                              long long s_unit, uint64_t* bar, uint64_t pol) {
  constexpr int BOX = tile_box_cols(BV);
#pragma unroll
  for (int b = 0; b < BV / BOX; ++b)
    tma_load_2d(tile + b * K * BOX, map, vt * BV + b * BOX, static_cast<int>(s_unit * K), bar, pol);
}

struct Item {
  int n, hv, h, vt;
  long long unit;    // n * HV + hv
  long long s_unit;  // state-pool slot * HV + hv: the item's S0 tile row / K
  long long cs_row;  // conv_state-pool slot
  long long im_row;  // inter_ssm / conv_snapshots-pool slot
  bool skip;         // padding sequence or out-of-range slot: touch nothing
  bool bad;          // out-of-range slot (reported in the status word)
};

__device__ __forceinline__ int resolve_slot(const int* idx, int n, int pool, bool& skip, bool& bad) {
  if (!idx) return n;
  const int sl = __ldg(idx + n);
  if (sl < 0) skip = true;
  if (sl >= pool) skip = bad = true;
  return sl;
}

// Items number fewer than 2^31 (N * HV * K < 2^31 is checked on the host and
// V / BV <= 16), so the decode divides in 32 bits.
__device__ __forceinline__ Item decode_item(const Params& p, long long item) {
  Item it;
  const uint32_t i32 = static_cast<uint32_t>(item);
  const uint32_t unit = fdiv(i32, p.div_nvt);
  const uint32_t n = fdiv(unit, p.div_HV);
  it.unit = unit;
  it.vt = static_cast<int>(i32 - unit * static_cast<uint32_t>(p.nvt));
  it.n = static_cast<int>(n);
  it.hv = static_cast<int>(unit - n * static_cast<uint32_t>(p.HV));
  it.h = static_cast<int>(fdiv(static_cast<uint32_t>(it.hv), p.div_G));
  it.skip = it.bad = false;
  const int ss = resolve_slot(p.idx_state, it.n, p.pool_state, it.skip, it.bad);
  const int cs = resolve_slot(p.idx_conv, it.n, p.pool_conv, it.skip, it.bad);
  const int im = resolve_slot(p.idx_inter, it.n, p.pool_inter, it.skip, it.bad);
  it.s_unit = (long long)ss * p.HV + it.hv;
  it.cs_row = cs;
  it.im_row = im;
  return it;
}

// First channel (within dim) of a block: kind 0 = q of head h, 1 = k of head
// h, 2 = the item's v tile.
template <int K, int BV>
__device__ __forceinline__ int block_channel(const Params& p, const Item& it, int kind) {
  return kind == 0 ? it.h * K
                   : (kind == 1 ? p.H * K + it.h * K : 2 * p.H * K + it.hv * p.V + it.vt * BV);
}

// ---------------------------------------------------------------------------
// where a producer task reads its raw inputs from; e0 = first channel of an
// 8-(bf16) / 4-(fp32) channel vector within the block
// ---------------------------------------------------------------------------

// Straight from global memory (one-item-per-CTA kernel).
template <typename Act, int K, int BV>
struct GlobalSrc {
  const Params& p;
  const Item& it;
  __device__ __forceinline__ uint4 x(int kind, int t, int e0) const {
    const Act* b = static_cast<const Act*>(p.mixed_qkv) + ((size_t)it.n * p.T + t) * p.dim;
    return ld_ro_16(b + block_channel<K, BV>(p, it, kind) + e0);
  }
  __device__ __forceinline__ uint4 cs(int kind, int e0, int m) const {
    const Act* b = static_cast<const Act*>(p.conv_state) +
                   ((size_t)it.cs_row * p.dim + block_channel<K, BV>(p, it, kind) + e0) * (kConvW - 1);
    return ld_rw_16(reinterpret_cast<const char*>(b) + 16 * m);
  }
  __device__ __forceinline__ uint4 w(int kind, int e0, int m) const {
    const Act* b = static_cast<const Act*>(p.conv_w) +
                   (size_t)(block_channel<K, BV>(p, it, kind) + e0) * kConvW;
    return ld_ro_16(reinterpret_cast<const char*>(b) + 16 * m);
  }
  __device__ __forceinline__ uint4 a(int t, int e0) const {
    return ld_ro_16(static_cast<const Act*>(p.a) + (((size_t)it.n * p.T + t) * p.HV + it.hv) * K + e0);
  }
  __device__ __forceinline__ float4 dt(int e0) const {
    return __ldg(reinterpret_cast<const float4*>(p.dt_bias + (size_t)it.hv * K + e0));
  }
};

// From an item's raw inputs staged in shared memory by 1-D bulk copies (the
// pipelined kernel); same interface as GlobalSrc.
template <typename Act, int K, int BV>
struct SmemSrc {
  const unsigned char* raw;
  int T;
  static constexpr int AB = sizeof(Act);
  // x_q [T][K] | x_k [T][K] | x_v [T][BV] | cs [2K+BV][3] | w [2K+BV][4] | a [T][K] | dt [K]
  __device__ __forceinline__ size_t off_x(int kind, int t) const {
    return kind == 0 ? (size_t)t * K * AB
                     : (kind == 1 ? (size_t)(T + t) * K * AB
                                  : (size_t)2 * T * K * AB + (size_t)t * BV * AB);
  }
  __device__ __forceinline__ size_t base_cs() const { return (size_t)T * (2 * K + BV) * AB; }
  __device__ __forceinline__ size_t base_w() const { return base_cs() + (size_t)(2 * K + BV) * 3 * AB; }
  __device__ __forceinline__ size_t base_a() const { return base_w() + (size_t)(2 * K + BV) * 4 * AB; }
  __device__ __forceinline__ size_t base_dt() const { return base_a() + (size_t)T * K * AB; }
  __device__ __forceinline__ static int blk(int kind) { return kind == 0 ? 0 : (kind == 1 ? K : 2 * K); }
  __device__ __forceinline__ uint4 x(int kind, int t, int e0) const {
    return *reinterpret_cast<const uint4*>(raw + off_x(kind, t) + (size_t)e0 * AB);
  }
  __device__ __forceinline__ uint4 cs(int kind, int e0, int m) const {
    return *reinterpret_cast<const uint4*>(raw + base_cs() + (size_t)(blk(kind) + e0) * 3 * AB + 16 * m);
  }
  __device__ __forceinline__ uint4 w(int kind, int e0, int m) const {
    return *reinterpret_cast<const uint4*>(raw + base_w() + (size_t)(blk(kind) + e0) * 4 * AB + 16 * m);
  }
  __device__ __forceinline__ uint4 a(int t, int e0) const {
    return *reinterpret_cast<const uint4*>(raw + base_a() + ((size_t)t * K + e0) * AB);
  }
  __device__ __forceinline__ float4 dt(int e0) const {
    return *reinterpret_cast<const float4*>(raw + base_dt() + (size_t)e0 * 4);
  }
};

// bytes of one item's staged raw inputs (SmemSrc layout; dt only with the
// softplus gate, but always reserved)
__host__ __device__ constexpr size_t raw_bytes(int T, int K, int BV, int ab) {
  return (size_t)ab * ((size_t)T * (2 * K + BV) + (size_t)(2 * K + BV) * 7 + (size_t)T * K) +
         4 * (size_t)K;
}

// ---------------------------------------------------------------------------
// producer arithmetic (shared by both kernels)
// ---------------------------------------------------------------------------

// A producer thread's one-off work that needs no producer result (the state
// tile's barrier and TMA load, an L2 prefetch of a later item): run once per
// thread right after the global loads of its first task are issued and before
// their values are used, so the ~0.5-1 us that issuing it holds the thread
// overlaps those loads' latency instead of delaying them.
struct NoHook {
  __device__ __forceinline__ void operator()() const {}
};

// Select x_ext[idx] (idx < 3: the old state) with compile-time register
// indices only.
template <typename Raw, int VEC>
__device__ __forceinline__ void select_state(const Raw (&cs)[3 * VEC], int idx, Raw (&out)[VEC]) {
#pragma unroll
  for (int jj = 0; jj < kConvW - 1; ++jj)
    if (jj == idx) {
#pragma unroll
      for (int e = 0; e < VEC; ++e) out[e] = cs[e * (kConvW - 1) + jj];
    }
}

// One conv task: VEC channels of block `kind` at token t.  Writes SiLU(conv)
// to y[e], the snapshot of token t when `snap`, at t = T-1 the rolled state of
// these channels when `roll`, and the raw window after token t (three 16-byte
// words) to `stash` when it is not null.  This form unpacks every input value
// into its own register (fewest instructions); conv_task_packed below does the
// same arithmetic from packed words, for kernels with a tight register cap.
template <typename Act, typename Src, typename Hook = NoHook>
__device__ __forceinline__ void conv_task_unpacked(const Src& src, const Params& p, const Item& it,
                                          int kind, int e0, int c, int t,
                                          float (&y)[ActT<Act>::VEC], bool snap, bool roll,
                                          uint4* stash, const Hook* hook = nullptr) {
  using AT = ActT<Act>;
  using Raw = typename AT::Raw;
  constexpr int VEC = AT::VEC;
  const int T = p.T;
  Raw cs[3 * VEC] = {};
  Raw win[kConvW][VEC];  // window x_ext[t .. t+3]: x_ext[i] = state[i] for i < 3, else token i-3
  Raw wr[4 * VEC];
  if constexpr (std::is_same<Hook, NoHook>::value) {
    // unpack each word as it is loaded (fewest live registers)
    if (t < kConvW - 1) {
#pragma unroll
      for (int m = 0; m < 3; ++m) AT::unpack(src.cs(kind, e0, m), cs + m * VEC);
    }
#pragma unroll
    for (int j = 0; j < kConvW; ++j) {
      const int idx = t + j;
      if (idx >= kConvW - 1) AT::unpack(src.x(kind, idx - (kConvW - 1), e0), win[j]);
      else select_state<Raw, VEC>(cs, idx, win[j]);
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) AT::unpack(src.w(kind, e0, m), wr + m * VEC);
  } else {
    // every load first, the hook while they are in flight, then unpack
    uint4 csw[3] = {};
    if (t < kConvW - 1) {
#pragma unroll
      for (int m = 0; m < 3; ++m) csw[m] = src.cs(kind, e0, m);
    }
    uint4 xw[kConvW] = {};
#pragma unroll
    for (int j = 0; j < kConvW; ++j)
      if (t + j >= kConvW - 1) xw[j] = src.x(kind, t + j - (kConvW - 1), e0);
    uint4 ww[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) ww[m] = src.w(kind, e0, m);
    if (hook) (*hook)();
    if (t < kConvW - 1) {
#pragma unroll
      for (int m = 0; m < 3; ++m) AT::unpack(csw[m], cs + m * VEC);
    }
#pragma unroll
    for (int j = 0; j < kConvW; ++j) {
      const int idx = t + j;
      if (idx >= kConvW - 1) AT::unpack(xw[j], win[j]);
      else select_state<Raw, VEC>(cs, idx, win[j]);
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) AT::unpack(ww[m], wr + m * VEC);
  }
#pragma unroll
  for (int e = 0; e < VEC; ++e) {
    float acc = __fmul_rn(AT::to_f(wr[e * kConvW]), AT::to_f(win[0][e]));
#pragma unroll
    for (int j = 1; j < kConvW; ++j) acc = __fmaf_rn(AT::to_f(wr[e * kConvW + j]), AT::to_f(win[j][e]), acc);
    y[e] = silu_f(acc);
  }
  const bool do_roll = roll && t == T - 1;
  if (snap || do_roll || stash) {
    // the raw window after token t: x_ext[t+1 .. t+3], channel-major [e][j]
    Raw r[3 * VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e)
#pragma unroll
      for (int j = 0; j < kConvW - 1; ++j) r[e * (kConvW - 1) + j] = win[j + 1][e];
    if (snap) {
      char* sp = reinterpret_cast<char*>(static_cast<Act*>(p.conv_snapshots) +
                                         (((size_t)it.im_row * T + t) * p.dim + c) * (kConvW - 1));
#pragma unroll
      for (int m = 0; m < 3; ++m) st_16(sp + 16 * m, AT::pack(r + m * VEC));
    }
    if (do_roll) {
      char* cp = reinterpret_cast<char*>(static_cast<Act*>(p.conv_state) +
                                         ((size_t)it.cs_row * p.dim + c) * (kConvW - 1));
#pragma unroll
      for (int m = 0; m < 3; ++m) st_16(cp + 16 * m, AT::pack(r + m * VEC));
    }
    if (stash) {
#pragma unroll
      for (int m = 0; m < 3; ++m) stash[m] = AT::pack(r + m * VEC);
    }
  }
}

// Raw value i (compile-time after unrolling) of a 16-byte word of
// activations: 8 bf16 halves or 4 fp32 words.
template <typename Act>
__device__ __forceinline__ uint32_t raw_at(const uint4& w, int i) {
  if constexpr (sizeof(Act) == 4) {
    return i == 0 ? w.x : (i == 1 ? w.y : (i == 2 ? w.z : w.w));
  } else {
    const int q = i >> 1;
    const uint32_t word = q == 0 ? w.x : (q == 1 ? w.y : (q == 2 ? w.z : w.w));
    return (i & 1) ? (word >> 16) : (word & 0xffffu);
  }
}

// The conv task of conv_task_unpacked with its inputs kept packed in 16-byte
// words
// (window positions, the old state [e][j], the taps [e][j]) and single values
// are extracted where they are used.
template <typename Act, typename Src, typename Hook = NoHook>
__device__ __forceinline__ void conv_task_packed(const Src& src, const Params& p, const Item& it,
                                          int kind, int e0, int c, int t,
                                          float (&y)[ActT<Act>::VEC], bool snap, bool roll,
                                          uint4* stash, const Hook* hook = nullptr) {
  using AT = ActT<Act>;
  using Raw = typename AT::Raw;
  constexpr int VEC = AT::VEC;
  const int T = p.T;
  uint4 csw[3] = {};
  if (t < kConvW - 1) {
#pragma unroll
    for (int m = 0; m < 3; ++m) csw[m] = src.cs(kind, e0, m);
  }
  // window x_ext[t .. t+3]: x_ext[i] = state[i] for i < 3, else token i-3
  uint4 xw[kConvW] = {};
#pragma unroll
  for (int j = 0; j < kConvW; ++j)
    if (t + j >= kConvW - 1) xw[j] = src.x(kind, t + j - (kConvW - 1), e0);
  // raw value of channel e at window position j
  auto xraw = [&](int j, int e) -> Raw {
    const int idx = t + j;
    if (idx >= kConvW - 1) return raw_at<Act>(xw[j], e);
    const Raw s0 = raw_at<Act>(csw[(e * 3 + 0) / VEC], (e * 3 + 0) % VEC);
    const Raw s1 = raw_at<Act>(csw[(e * 3 + 1) / VEC], (e * 3 + 1) % VEC);
    const Raw s2 = raw_at<Act>(csw[(e * 3 + 2) / VEC], (e * 3 + 2) % VEC);
    return idx == 0 ? s0 : (idx == 1 ? s1 : s2);
  };
  uint4 ww[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) ww[m] = src.w(kind, e0, m);
  if (hook) (*hook)();
#pragma unroll
  for (int e = 0; e < VEC; ++e) {
    float acc = __fmul_rn(AT::to_f(raw_at<Act>(ww[(e * 4) / VEC], (e * 4) % VEC)), AT::to_f(xraw(0, e)));
#pragma unroll
    for (int j = 1; j < kConvW; ++j)
      acc = __fmaf_rn(AT::to_f(raw_at<Act>(ww[(e * 4 + j) / VEC], (e * 4 + j) % VEC)),
                      AT::to_f(xraw(j, e)), acc);
    y[e] = silu_f(acc);
  }
  const bool do_roll = roll && t == T - 1;
  if (snap || do_roll || stash) {
    // the raw window after token t: x_ext[t+1 .. t+3], channel-major [e][j]
    Raw r[3 * VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e)
#pragma unroll
      for (int j = 0; j < kConvW - 1; ++j) r[e * (kConvW - 1) + j] = xraw(j + 1, e);
    if (snap) {
      char* sp = reinterpret_cast<char*>(static_cast<Act*>(p.conv_snapshots) +
                                         (((size_t)it.im_row * T + t) * p.dim + c) * (kConvW - 1));
#pragma unroll
      for (int m = 0; m < 3; ++m) st_16(sp + 16 * m, AT::pack(r + m * VEC));
    }
    if (do_roll) {
      char* cp = reinterpret_cast<char*>(static_cast<Act*>(p.conv_state) +
                                         ((size_t)it.cs_row * p.dim + c) * (kConvW - 1));
#pragma unroll
      for (int m = 0; m < 3; ++m) st_16(cp + 16 * m, AT::pack(r + m * VEC));
    }
    if (stash) {
#pragma unroll
      for (int m = 0; m < 3; ++m) stash[m] = AT::pack(r + m * VEC);
    }
  }
}

// The raw inputs of one gate task (VEC channels at token t): the gate logits
// and, with the softplus gate, dt_bias.
template <typename Act>
struct GateIn {
  uint4 a;
  float4 dt[ActT<Act>::VEC / 4];
};

template <typename Act, typename Src>
__device__ __forceinline__ GateIn<Act> gate_load(const Src& src, int gate_mode, int t, int e0) {
  GateIn<Act> g;
  g.a = src.a(t, e0);
  if (gate_mode == 0) {
#pragma unroll
    for (int e = 0; e < ActT<Act>::VEC; e += 4) g.dt[e / 4] = src.dt(e0 + e);
  }
  return g;
}

// alpha = exp(g) of a gate task's VEC channels.
template <typename Act>
__device__ __forceinline__ void gate_math(const GateIn<Act>& in, int gate_mode, float negA,
                                          float (&al)[ActT<Act>::VEC]) {
  using AT = ActT<Act>;
  using Raw = typename AT::Raw;
  constexpr int VEC = AT::VEC;
  Raw r[VEC];
  AT::unpack(in.a, r);
  if (gate_mode == 0) {
#pragma unroll
    for (int e = 0; e < VEC; e += 4) {
      const float4 d = in.dt[e / 4];
      const float dd[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float x = __fadd_rn(AT::to_f(r[e + j]), dd[j]);
        al[e + j] = decay_f(__fmul_rn(negA, softplus_f(x)));
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < VEC; ++e) al[e] = decay_f(fminf(AT::to_f(r[e]), 0.0f));
  }
}

// One gate task: alpha = exp(g) of VEC channels at token t.
template <typename Act, typename Src>
__device__ __forceinline__ void gate_task(const Src& src, int gate_mode, float negA, int t,
                                          int e0, float (&al)[ActT<Act>::VEC]) {
  gate_math<Act>(gate_load<Act>(src, gate_mode, t, e0), gate_mode, negA, al);
}

template <typename Act>
__device__ __forceinline__ float load_b(const Params& p, const Item& it, int t) {
  const Act* bp = static_cast<const Act*>(p.b) + ((size_t)it.n * p.T + t) * p.HV + it.hv;
  if constexpr (sizeof(Act) == 4) {
    return __ldg(reinterpret_cast<const float*>(bp));
  } else {
    return ActT<Act>::to_f(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(bp))));
  }
}

// All conv / gate / beta tasks of one item, spread over `nthr` threads.
// With `stash` null the v tile's conv_state is rolled here (its raw inputs
// already sit in shared memory, so no reader is left in global memory);
// otherwise the raw window after the last token of every channel vector cv is
// staged at stash[3 cv .. 3 cv + 2] and the caller rolls after a barrier.
// ext_b / ext_negA, when not null, hold this item's beta logits b[t] and
// -exp(A_log[hv]) (loaded ahead by the caller); otherwise they are read here.
template <typename Act, int K, int BV, bool DEC = false, bool PACKED = false, typename Src,
          typename Hook = NoHook>
__device__ __forceinline__ void produce_tasks(const Src& src, const Params& p, const Item& it,
                                              float* sQ, float* sK, float* sA, float* sV,
                                              float* sB, uint4* stash, int tid, int nthr,
                                              const float* ext_b = nullptr,
                                              const float* ext_negA = nullptr,
                                              const Hook& hook = Hook()) {
  constexpr int VEC = ActT<Act>::VEC;
  constexpr int NQ = K / VEC;
  constexpr int NCV = 2 * NQ + BV / VEC;  // channel vectors of the item
  constexpr int KS = stage_ks(K);
  const int T = p.T;
  const int n_conv = NCV * T;
  const int n_gate = NQ * T;
  // q/k snapshots are written once per group: by its first v-head, first tile
  const bool qk_snap_owner = !DEC && (it.hv == it.h * p.G) && (it.vt == 0);
  constexpr bool v_snap = !DEC;  // decode writes no conv-window snapshots
  // Beta of token t rides on the gate task of its first channel vector.  When
  // the threads outnumber the tasks, the gate tasks start on a warp boundary,
  // so that no warp runs the conv and the gate code paths one after the
  // other: the producer's latency is the longer path, not the sum.
  const int gate0 = (n_conv + 31) & ~31;
  const bool spread = gate0 + n_gate <= nthr;
  const int n_slots = spread ? gate0 + n_gate : n_conv + n_gate;
  // the hook runs in this thread's first task (after its loads) or, with no
  // task, after the loop
  const bool has_task = tid < n_slots && !(spread && tid >= n_conv && tid < gate0);
  if (!has_task) hook();
  for (int slot = tid; slot < n_slots; slot += nthr) {
    int task = slot;
    if (spread && slot >= n_conv) {
      if (slot < gate0) continue;  // padding up to a warp boundary
      task = n_conv + (slot - gate0);
    }
    const Hook* hk = slot == tid ? &hook : nullptr;
    if (task < n_conv) {
      const int cv = static_cast<int>(fdiv(static_cast<uint32_t>(task), p.div_T));
      const int t = task - cv * T;
      const int kind = cv < NQ ? 0 : (cv < 2 * NQ ? 1 : 2);
      const int e0 = (cv - kind * NQ) * VEC;
      const int c = block_channel<K, BV>(p, it, kind) + e0;
      float y[VEC];
      const bool roll_v = kind == 2 && !stash;
      uint4* st = (stash && t == T - 1) ? stash + 3 * cv : nullptr;
      if constexpr (PACKED)
        conv_task_packed<Act>(src, p, it, kind, e0, c, t, y, kind == 2 ? v_snap : qk_snap_owner, roll_v, st, hk);
      else
        conv_task_unpacked<Act>(src, p, it, kind, e0, c, t, y, kind == 2 ? v_snap : qk_snap_owner, roll_v, st, hk);
      if (kind == 2) {  // v: column order
#pragma unroll
        for (int e = 0; e < VEC; e += 4)
          *reinterpret_cast<float4*>(sV + t * BV + e0 + e) = make_float4(y[e], y[e + 1], y[e + 2], y[e + 3]);
      } else {  // q, k: the consumers' row order
        float* dst = (kind == 0 ? sQ : sK) + t * KS;
#pragma unroll
        for (int e = 0; e < VEC; ++e) dst[stage_pos<K>(e0 + e)] = y[e];
      }
    } else {
      const int g = task - n_conv;
      const int t = g / NQ;
      const int e0 = (g - t * NQ) * VEC;
      // every load first (the hook runs while they are in flight), then the math
      const float braw = e0 == 0 ? (ext_b ? ext_b[t] : load_b<Act>(p, it, t)) : 0.0f;
      const float alog = (p.gate_mode != 0 || ext_negA) ? 0.0f : __ldg(p.A_log + it.hv);
      const GateIn<Act> gin = gate_load<Act>(src, p.gate_mode, t, e0);
      if (hk) (*hk)();
      const float negA = p.gate_mode != 0 ? 0.0f : (ext_negA ? *ext_negA : -expf(alog));
      float al[VEC];
      gate_math<Act>(gin, p.gate_mode, negA, al);
#pragma unroll
      for (int e = 0; e < VEC; ++e) sA[t * KS + stage_pos<K>(e0 + e)] = al[e];
      if (e0 == 0) sB[t] = sigmoid_f(braw);
    }
  }
}

// L2 norm of one staged K-vector by one warp (q additionally scaled by
// K^-1/2); lane l takes channels l, l + 32, ...
template <int K>
__device__ __forceinline__ void l2norm_warp(float* x, bool is_q, int lane) {
  float xs[K / 32];
  float ss = 0.0f;
#pragma unroll
  for (int m = 0; m < K / 32; ++m) {
    xs[m] = x[stage_pos<K>(lane + 32 * m)];
    ss = __fmaf_rn(xs[m], xs[m], ss);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
  float inv = rsqrtf(__fadd_rn(ss, kL2Eps));
  if (is_q) inv = __fmul_rn(inv, rsqrtf(static_cast<float>(K)));
#pragma unroll
  for (int m = 0; m < K / 32; ++m) x[stage_pos<K>(lane + 32 * m)] = __fmul_rn(xs[m], inv);
}

// Store the staged windows x_ext[T .. T+2] (produce_tasks' stash) of channel
// vectors [cv0, cv1) as the new conv_state: the q/k blocks are vectors
// [0, 2K/VEC), the item's v tile the rest.  Called after a barrier that
// follows every conv_state read of the CTA.
template <typename Act, int K, int BV>
__device__ __forceinline__ void roll_staged(const Params& p, const Item& it, const uint4* stash,
                                            int cv0, int cv1, int tid, int nthr) {
  constexpr int VEC = ActT<Act>::VEC;
  constexpr int NQ = K / VEC;
  for (int cv = cv0 + tid; cv < cv1; cv += nthr) {
    const int kind = cv < NQ ? 0 : (cv < 2 * NQ ? 1 : 2);
    const int c = block_channel<K, BV>(p, it, kind) + (cv - kind * NQ) * VEC;
    char* cp = reinterpret_cast<char*>(static_cast<Act*>(p.conv_state) +
                                       ((size_t)it.cs_row * p.dim + c) * (kConvW - 1));
#pragma unroll
    for (int m = 0; m < 3; ++m) st_16(cp + 16 * m, stash[3 * cv + m]);
  }
}

// ---------------------------------------------------------------------------
// consumer: the recurrence on register-resident S
// ---------------------------------------------------------------------------
template <int K, int BV>
__device__ __forceinline__ void load_tile(const float* sbuf, float4 (&s)[rows_per_thread(K)], int warp,
                                          int lane) {
  constexpr int R = rows_per_thread(K);
  constexpr int CQ = 32 / row_groups(K);
  const int rg = lane / CQ, cg = lane % CQ;
  const int col = warp * warp_cols(K) + cg * 4;
#pragma unroll
  for (int i = 0; i < R; ++i)
    s[i] = *reinterpret_cast<const float4*>(sbuf + tile_index<K, BV>(own_row<K>(rg, i), col));
}

template <typename Act, int K, int BV, bool DEC = false>
__device__ __forceinline__ void consume(const Params& p, const Item& it, const float* sQ,
                                       const float* sK, const float* sA, const float* sV,
                                       const float* sB, float4 (&s)[rows_per_thread(K)], int warp,
                                       int lane) {
  constexpr int R = rows_per_thread(K);
  constexpr int CQ = 32 / row_groups(K);
  constexpr int RS = stage_rs(K);
  constexpr int KS = stage_ks(K);
  const int rg = lane / CQ;
  const int cg = lane % CQ;
  const int col = warp * warp_cols(K) + cg * 4;  // column within the tile
  const int T = p.T;
  const int V = p.V;
  const size_t colg = (size_t)it.vt * BV + col;  // column within the state
  for (int t = 0; t < T; ++t) {
    const float* al = sA + t * KS + rg * RS;
    const float* kk = sK + t * KS + rg * RS;
    const float* qq = sQ + t * KS + rg * RS;
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
    for (int off = CQ; off <= 16; off <<= 1) {
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
    // this thread's rows are own_row(rg, i) = RG i + row_perm(rg): start at
    // row row_perm(rg), step RG rows
    float* dst = DEC ? nullptr
                     : p.inter_ssm + ((((size_t)it.im_row * T + t) * p.HV + it.hv) * K + row_perm<K>(rg)) * V + colg;
    const size_t step8 = (size_t)row_groups(K) * V;
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
        if constexpr (!DEC) st_stream_f4(dst + (size_t)(i + j) * step8, x);
      }
    }
#pragma unroll
    for (int off = CQ; off <= 16; off <<= 1) {
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
  if constexpr (DEC) {
    // decode: the state after the last token replaces the persistent state
    float* dst = p.S_out + ((size_t)it.s_unit * K + row_perm<K>(rg)) * V + colg;
#pragma unroll
    for (int i = 0; i < R; ++i) st_stream_f4(dst + (size_t)i * row_groups(K) * V, s[i]);
  }
}

// L2 prefetch of everything item `itm` reads from HBM: its state tile and its
// raw input rows (q/k/v token rows, conv_state blocks, gate rows), spread over
// the lanes of one warp.  Issued about one residency wave ahead, so the CTA
// that later takes the item finds its inputs in L2.
template <typename Act, int K, int BV>
__device__ __forceinline__ void prefetch_item_l2(const Params& p, const CUtensorMap* tmap,
                                                 long long itm, int lane) {
  constexpr int AB = sizeof(Act);
  const Item it = decode_item(p, itm);
  if (it.skip) return;
  const int T = p.T;
  const int n_pf = 3 * T + 3 + T + 1;
  for (int c = lane; c < n_pf; c += 32) {
    if (c < 3 * T) {
      const int t = c / 3, kind = c - 3 * t;
      const char* src = static_cast<const char*>(p.mixed_qkv) +
                        (((size_t)it.n * T + t) * p.dim + block_channel<K, BV>(p, it, kind)) * AB;
      bulk_prefetch_l2(src, (kind == 2 ? BV : K) * AB);
    } else if (c < 3 * T + 3) {
      const int kind = c - 3 * T;
      const char* src = static_cast<const char*>(p.conv_state) +
                        ((size_t)it.cs_row * p.dim + block_channel<K, BV>(p, it, kind)) * 3 * AB;
      bulk_prefetch_l2(src, (kind == 2 ? BV : K) * 3 * AB);
    } else if (c < 4 * T + 3) {
      const int t = c - 3 * T - 3;
      bulk_prefetch_l2(static_cast<const char*>(p.a) +
                           ((((size_t)it.n * T + t) * p.HV + it.hv) * K) * AB,
                       K * AB);
    } else {
      constexpr int BOX = tile_box_cols(BV);
#pragma unroll
      for (int bx = 0; bx < BV / BOX; ++bx)
        tma_prefetch_2d(tmap, it.vt * BV + bx * BOX, static_cast<int>(it.s_unit * K));
    }
  }
}

// The same recurrence with S kept in the shared-memory tile instead of
// registers (about half the registers, so more CTAs per SM).  Each thread
// owns exactly the elements the register consumer holds; per token, pass 1
// decays them and forms the partial S^T k, pass 2 recomputes the decayed
// value (the same fmul, hence the same bits), applies the rank-1 update, forms
// the partial S^T q, stores the snapshot and writes the element back.  The
// floating-point operations and their order are those of `consume`, so the
// results are bit-identical.
template <typename Act, int K, int BV, bool DEC = false>
__device__ __forceinline__ void consume_smem(const Params& p, const Item& it, const float* sQ,
                                            const float* sK, const float* sA, const float* sV,
                                            const float* sB, float* sS, int warp, int lane) {
  constexpr int R = rows_per_thread(K);
  constexpr int CQ = 32 / row_groups(K);
  constexpr int RS = stage_rs(K);
  constexpr int KS = stage_ks(K);
  const int rg = lane / CQ;
  const int cg = lane % CQ;
  const int col = warp * warp_cols(K) + cg * 4;
  const int T = p.T;
  const int V = p.V;
  const size_t colg = (size_t)it.vt * BV + col;

  for (int t = 0; t < T; ++t) {
    const float* al = sA + t * KS + rg * RS;
    const float* kk = sK + t * KS + rg * RS;
    const float* qq = sQ + t * KS + rg * RS;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < R; i += 4) {
      const float4 a4 = *reinterpret_cast<const float4*>(al + i);
      const float4 k4 = *reinterpret_cast<const float4*>(kk + i);
      const float av[4] = {a4.x, a4.y, a4.z, a4.w};
      const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float4 x = *reinterpret_cast<const float4*>(sS + tile_index<K, BV>(own_row<K>(rg, i + j), col));
        x.x = __fmul_rn(x.x, av[j]); x.y = __fmul_rn(x.y, av[j]);
        x.z = __fmul_rn(x.z, av[j]); x.w = __fmul_rn(x.w, av[j]);
        acc.x = __fmaf_rn(x.x, kv[j], acc.x); acc.y = __fmaf_rn(x.y, kv[j], acc.y);
        acc.z = __fmaf_rn(x.z, kv[j], acc.z); acc.w = __fmaf_rn(x.w, kv[j], acc.w);
      }
    }
#pragma unroll
    for (int off = CQ; off <= 16; off <<= 1) {
      acc.x = __fadd_rn(acc.x, __shfl_xor_sync(0xffffffffu, acc.x, off));
      acc.y = __fadd_rn(acc.y, __shfl_xor_sync(0xffffffffu, acc.y, off));
      acc.z = __fadd_rn(acc.z, __shfl_xor_sync(0xffffffffu, acc.z, off));
      acc.w = __fadd_rn(acc.w, __shfl_xor_sync(0xffffffffu, acc.w, off));
    }
    const float4 v4 = *reinterpret_cast<const float4*>(sV + t * BV + col);
    const float be = sB[t];
    float4 u;
    u.x = __fmul_rn(be, __fsub_rn(v4.x, acc.x)); u.y = __fmul_rn(be, __fsub_rn(v4.y, acc.y));
    u.z = __fmul_rn(be, __fsub_rn(v4.z, acc.z)); u.w = __fmul_rn(be, __fsub_rn(v4.w, acc.w));
    const bool last = t == T - 1;
    float* dst = DEC ? (last ? p.S_out + ((size_t)it.s_unit * K + row_perm<K>(rg)) * V + colg : nullptr)
                     : p.inter_ssm + ((((size_t)it.im_row * T + t) * p.HV + it.hv) * K + row_perm<K>(rg)) * V + colg;
    const size_t step8 = (size_t)row_groups(K) * V;
    float4 oa = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < R; i += 4) {
      const float4 a4 = *reinterpret_cast<const float4*>(al + i);
      const float4 k4 = *reinterpret_cast<const float4*>(kk + i);
      const float4 q4 = *reinterpret_cast<const float4*>(qq + i);
      const float av[4] = {a4.x, a4.y, a4.z, a4.w};
      const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
      const float qv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float4* ep = reinterpret_cast<float4*>(sS + tile_index<K, BV>(own_row<K>(rg, i + j), col));
        float4 x = *ep;
        x.x = __fmul_rn(x.x, av[j]); x.y = __fmul_rn(x.y, av[j]);
        x.z = __fmul_rn(x.z, av[j]); x.w = __fmul_rn(x.w, av[j]);
        x.x = __fmaf_rn(kv[j], u.x, x.x); x.y = __fmaf_rn(kv[j], u.y, x.y);
        x.z = __fmaf_rn(kv[j], u.z, x.z); x.w = __fmaf_rn(kv[j], u.w, x.w);
        oa.x = __fmaf_rn(x.x, qv[j], oa.x); oa.y = __fmaf_rn(x.y, qv[j], oa.y);
        oa.z = __fmaf_rn(x.z, qv[j], oa.z); oa.w = __fmaf_rn(x.w, qv[j], oa.w);
        if (DEC ? last : true) st_stream_f4(dst + (size_t)(i + j) * step8, x);
        if (!last) *ep = x;
      }
    }
#pragma unroll
    for (int off = CQ; off <= 16; off <<= 1) {
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
// split variant: the stage of an item travels from the prep kernel to the
// recurrence kernel inside the item's own snapshot of the last token
// ---------------------------------------------------------------------------
// The stage (q, k, alpha [T][KS], v [T][BV], beta [round4(T)], the layout the
// consumer reads) is kept in the first rows of the K x BV slice that the item
// later overwrites with its state after token T-1: stage float s at row
// s / BV, column s % BV.  The item's CTA reads it all into shared memory
// before a barrier and only then writes any snapshot.  The host checks that
// stage_floats(T, K, BV) <= K * BV.
template <int K, int BV>
__device__ __forceinline__ float* stage_home(const Params& p, const Item& it) {
  return p.inter_ssm + (((size_t)it.im_row * p.T + p.T - 1) * p.HV + it.hv) * (size_t)K * p.V +
         (size_t)it.vt * BV;
}

// Copy the item's stage from its home into shared memory (16-byte pieces).
template <int K, int BV>
__device__ __forceinline__ void copy_stage_in(const Params& p, const Item& it, float* stage, int tid,
                                              int nthr) {
  const float* home = stage_home<K, BV>(p, it);
  const int n4 = stage_floats(p.T, K, BV) / 4;
  for (int i = tid; i < n4; i += nthr) {
    const int sidx = 4 * i;
    *reinterpret_cast<float4*>(stage + sidx) =
        __ldcg(reinterpret_cast<const float4*>(home + (size_t)(sidx / BV) * p.V + (sidx % BV)));
  }
}

// L2 prefetch of item `itm`'s state tile only (the recurrence kernel of the
// split variant reads no raw inputs).
template <int K, int BV>
__device__ __forceinline__ void prefetch_tile_l2(const Params& p, const CUtensorMap* tmap, long long itm,
                                                 int lane) {
  constexpr int BOX = tile_box_cols(BV);
  const Item it = decode_item(p, itm);
  if (it.skip) return;
  for (int bx = lane; bx < BV / BOX; bx += 32)
    tma_prefetch_2d(tmap, it.vt * BV + bx * BOX, static_cast<int>(it.s_unit * K));
}

// ---------------------------------------------------------------------------
// one item per CTA: every warp produces, then consumes
// ---------------------------------------------------------------------------
// SMS: keep S in the shared-memory tile (consume_smem) instead of registers;
// the register cap then allows 3 CTAs of 8 warps per SM.
__host__ __device__ constexpr int tile_min_blocks(int warps, bool sms) {
  return sms ? 24 / warps : 16 / warps;
}

// PRE: the recurrence kernel of the split variant -- the stage comes from the
// prep kernel (through the item's home), which also wrote the conv snapshots
// and rolled the conv_state; launched as its programmatic dependent, the CTA
// issues its state-tile load before waiting for the prep kernel.
// RM, who rolls a q/k conv_state that several items read:
//   kRollCounter  the last arrival on the group's counter, or the separate
//                 roll kernel (Params::qk_roll_kernel), chosen at launch;
//   kRollCluster  launched as clusters of the G * nvt items of one q/k group:
//                 every CTA arrives on the cluster barrier once its
//                 conv_state reads are done, and the cluster's first CTA rolls
//                 the group's q/k conv_state after the wait;
//   kRollNone     no counter in the kernel: one reader per group (which rolls
//                 itself) or the separate roll kernel.  The decode kernels use
//                 it where they can: without the counter's pointer and count
//                 held across the recurrence they keep every value in
//                 registers (3-5 % faster from three tokens on, measured).
constexpr int kRollCounter = 0, kRollCluster = 1, kRollNone = 2;

template <typename Act, int K, int WARPS, bool DEC = false, bool SMS = false, bool PRE = false,
          int RM = kRollCounter>
__global__ void __launch_bounds__(WARPS * 32, tile_min_blocks(WARPS, SMS))
    kda_tile_kernel(const __grid_constant__ CUtensorMap tmap_s0, const Params p) {
  constexpr int BV = WARPS * warp_cols(K);
  constexpr int NT = WARPS * 32;
  constexpr int R = rows_per_thread(K);
  static_assert(K == 32 || K == 64 || K == 128 || K == 256, "unsupported K");

  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem);
  float* sbuf = tile_base(smem);
  const int T = p.T;
  constexpr int KS = stage_ks(K);
  float* sQ = sbuf + K * BV;
  float* sK = sQ + T * KS;
  float* sA = sK + T * KS;
  float* sV = sA + T * KS;
  float* sB = sV + T * BV;
  uint4* sRoll = reinterpret_cast<uint4*>(sB + round4(T));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const long long item = blockIdx.x;
  // This grid is itself launched as a programmatic dependent of the stream's
  // previous kernel, so its CTAs may be resident before that kernel has
  // ended: every global access, reads of the slot indices included, comes
  // after this wait (a no-op when nothing is in flight).  The split
  // recurrence's dependency is the prep kernel, waited for below.
  if constexpr (!PRE) asm volatile("griddepcontrol.wait;" ::: "memory");
  // A programmatic dependent launched after this grid (the q/k roll kernel,
  // or the next call) may be scheduled once every CTA has got here, by which
  // time the previous kernel has completed; it waits for this one's end.
  asm volatile("griddepcontrol.launch_dependents;");
  if (item >= p.num_items) return;
  const Item it = decode_item(p, item);
  if (it.skip) {  // padding sequence: nothing to read or write
    if (!PRE && it.bad && tid == 0 && it.hv == 0 && it.vt == 0) atomicOr(p.status, kStatusBadIndex);
    return;
  }

  // thread 0: the state tile's barrier and TMA load; the last warp: the L2
  // prefetch of a later item.  The register-state kernels run these as the
  // producer's hook, once each thread's first loads are in flight (measured
  // on GB300: 4-11 % faster over the 150-point sweep); the shared-memory-state
  // kernel, three CTAs per SM on short calls bound by the state traffic,
  // issues them first (the hook measured 3-12 % slower there).
  auto issue = [&]() {
    if (tid == 0) {
      mbar_init(mbar, 1);
      fence_mbar_init();
      prefetch_tensormap(&tmap_s0);
      mbar_arrive_expect_tx(mbar, K * BV * sizeof(float));
      tma_load_tile<K, BV>(sbuf, &tmap_s0, it.vt, it.s_unit, mbar, l2_policy_evict_first());
    }
    if (warp == WARPS - 1 && p.prefetch > 0 && item + p.prefetch < p.num_items) {
      if constexpr (PRE) prefetch_tile_l2<K, BV>(p, &tmap_s0, item + p.prefetch, lane);
      else prefetch_item_l2<Act, K, BV>(p, &tmap_s0, item + p.prefetch, lane);
    }
  };
  if constexpr (PRE || SMS) issue();
  if constexpr (PRE) {
    // the prep kernel has completed and its writes are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    copy_stage_in<K, BV>(p, it, sQ, tid, NT);
    __syncthreads();  // the stage is in shared memory before any snapshot overwrites its home
  } else {
    const GlobalSrc<Act, K, BV> src{p, it};
    if constexpr (SMS)
      produce_tasks<Act, K, BV, DEC, SMS>(src, p, it, sQ, sK, sA, sV, sB, sRoll, tid, NT);
    else
      produce_tasks<Act, K, BV, DEC, SMS>(src, p, it, sQ, sK, sA, sV, sB, sRoll, tid, NT, nullptr, nullptr,
                                          issue);
    __syncthreads();  // every conv_state read of this CTA is done, stage written
    // cluster protocol: this CTA's reads are done (their values are in shared
    // memory); the matching wait comes before the q/k roll at the end
    if constexpr (RM == kRollCluster) cluster_arrive_release();
    for (int r = warp; r < 2 * T; r += WARPS) l2norm_warp<K>(r < T ? sQ + r * KS : sK + (r - T) * KS, r < T, lane);
  }
  // Arrival on the q/k group counter by lane 0 of the last warp, after its
  // own rows (none while 2T < WARPS).  The returned count is first used at
  // the end of the CTA, so nothing waits here for the atomic's round trip.
  // With the separate roll kernel or the cluster there is no counter; in the
  // split variant the prep kernel rolls.
  constexpr int kRollWarp = WARPS - 1;
  const int expected = p.G * p.nvt;
  constexpr bool CL = RM == kRollCluster;
  const bool counted = !PRE && RM == kRollCounter && expected > 1 && !p.qk_roll_kernel;
  int* cnt = p.counters + (size_t)it.n * p.H + it.h;
  int arrival = 0;
  if (warp == kRollWarp && lane == 0 && counted) {
    __threadfence();  // the CTA's conv_state reads (before the barrier) come first
    arrival = atomicAdd(cnt, 1);
  }
  const bool ok = mbar_wait_bounded(mbar, 0, kWaitLimitNs);
  if (__syncthreads_or(!ok)) {
    // give up without hanging: report, keep the counter protocol intact, let
    // the copy in flight land, leave
    if (tid == 0) atomicOr(p.status, kStatusTmaTimeout);
    if (warp == kRollWarp && lane == 0 && counted && arrival == expected - 1) atomicExch(cnt, 0);
    mbar_wait_bounded(mbar, 0, kWaitLimitNs);
    if constexpr (CL) cluster_wait_acquire();  // every thread arrived before its own waits
    return;
  }
  if constexpr (SMS) {
    consume_smem<Act, K, BV, DEC>(p, it, sQ, sK, sA, sV, sB, sbuf, warp, lane);
  } else {
    float4 s[R];
    load_tile<K, BV>(sbuf, s, warp, lane);
    consume<Act, K, BV, DEC>(p, it, sQ, sK, sA, sV, sB, s, warp, lane);
  }
  if constexpr (PRE) return;
  constexpr int NQV = 2 * K / ActT<Act>::VEC;  // q/k channel vectors
  constexpr int NCV = NQV + BV / ActT<Act>::VEC;
  roll_staged<Act, K, BV>(p, it, sRoll, NQV, NCV, tid, NT);  // v: owned by this item
  // cluster: every CTA of the group has read its q/k conv_state once the wait
  // ends; rank 0 rolls
  if constexpr (CL) cluster_wait_acquire();
  if (warp == kRollWarp) {
    // q/k: the group's last arrival resets the counter and rolls
    const int last = __shfl_sync(0xffffffffu, expected == 1 || (counted && arrival == expected - 1) ||
                                                  (CL && cluster_cta_rank() == 0) ? 1 : 0, 0);
    if (last) {
      if (lane == 0 && counted) {
        atomicExch(cnt, 0);
        __threadfence();  // every other item's reads are ordered before the stores below
      }
      __syncwarp();
      roll_staged<Act, K, BV>(p, it, sRoll, 0, NQV, lane, 32);
    }
  }
}

// ---------------------------------------------------------------------------
// split variant, first kernel: the producer arithmetic of one q/k group
// ---------------------------------------------------------------------------
// One CTA per (sequence n, q/k head h): the conv + SiLU of the group's q and k
// channels and of the v channels of its G v-heads, their gates and betas, the
// q/k norms -- once per group instead of once per item that reads them; the
// conv snapshots and the rolled conv_state of all those channels (the group
// owns them: no other CTA reads them); then every item's stage (G v-heads x
// V / BV tiles), assembled from shared memory, written to its home.  The
// recurrence kernel, a programmatic dependent of this one, reads the stages.
constexpr int kPrepThreads = 256;

// floats of the prep kernel's shared staging: q, k [2][T][KS], alpha
// [G][T][KS], v [G][T][V], beta [G][round4(T)]; then the staged windows
__host__ __device__ constexpr size_t prep_stage_floats(int T, int K, int V, int G) {
  return (size_t)(2 + G) * T * stage_ks(K) + (size_t)G * T * V + (size_t)G * round4(T);
}
__host__ __device__ constexpr size_t prep_smem_bytes(int T, int K, int V, int G, int ab) {
  return sizeof(float) * prep_stage_floats(T, K, V, G) + (size_t)(2 * K + G * V) * 3 * ab;
}

template <typename Act, int K, int BV>
__global__ void __launch_bounds__(kPrepThreads) kda_prep_kernel(const Params p) {
  using AT = ActT<Act>;
  constexpr int VEC = AT::VEC;
  constexpr int NQ = K / VEC;  // q (or k) channel vectors
  constexpr int KS = stage_ks(K);
  const int T = p.T, G = p.G, V = p.V;
  const int NVV = V / VEC;     // v channel vectors of one v-head
  const int NCV = 2 * NQ + G * NVV;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  // launched as a programmatic dependent of the stream's previous kernel:
  // nothing global is touched before it has completed.  The recurrence
  // kernel, which issues its state-tile load before its own wait, may then be
  // scheduled once every CTA here has got past that wait.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int n = blockIdx.x / p.H;
  const int h = blockIdx.x - n * p.H;
  if (n >= p.N) return;
  // slots of sequence n from the group's first item
  const Item base = decode_item(p, ((long long)n * p.HV + (long long)h * G) * p.nvt);
  if (base.skip) {
    if (base.bad && h == 0 && tid == 0) atomicOr(p.status, kStatusBadIndex);
    return;
  }
  extern __shared__ __align__(128) unsigned char smem[];
  float* sQK = reinterpret_cast<float*>(smem);   // [2][T][KS]: q tokens, then k tokens
  float* sA = sQK + 2 * T * KS;                  // [G][T][KS]
  float* sV = sA + (size_t)G * T * KS;           // [G][T][V]
  float* sB = sV + (size_t)G * T * V;            // [G][round4(T)]
  uint4* stash = reinterpret_cast<uint4*>(sB + (size_t)G * round4(T));  // [NCV][3]

  // one task per (channel vector, token), then one per (v-head, 8 gate
  // channels, token); the gate tasks start on a warp boundary when the
  // threads outnumber the tasks (as in produce_tasks)
  const int n_conv = NCV * T;
  const int n_gate = G * NQ * T;
  const int gate0 = (n_conv + 31) & ~31;
  const bool spread = gate0 + n_gate <= kPrepThreads;
  const int n_slots = spread ? gate0 + n_gate : n_conv + n_gate;
  for (int slot = tid; slot < n_slots; slot += kPrepThreads) {
    int task = slot;
    if (spread && slot >= n_conv) {
      if (slot < gate0) continue;
      task = n_conv + (slot - gate0);
    }
    if (task < n_conv) {
      const int cv = static_cast<int>(fdiv(static_cast<uint32_t>(task), p.div_T));
      const int t = task - cv * T;
      const int kind = cv < NQ ? 0 : (cv < 2 * NQ ? 1 : 2);
      const int g = kind == 2 ? (cv - 2 * NQ) / NVV : 0;
      const int e0 = kind == 2 ? (cv - 2 * NQ - g * NVV) * VEC : (cv - kind * NQ) * VEC;
      Item itg = base;
      itg.hv = h * G + g;
      itg.vt = 0;
      const GlobalSrc<Act, K, BV> src{p, itg};
      const int c = block_channel<K, BV>(p, itg, kind) + e0;
      float y[VEC];
      conv_task_unpacked<Act>(src, p, itg, kind, e0, c, t, y, true, false,
                              t == T - 1 ? stash + 3 * cv : nullptr);
      if (kind == 2) {
        float* dst = sV + ((size_t)g * T + t) * V + e0;
#pragma unroll
        for (int e = 0; e < VEC; e += 4)
          *reinterpret_cast<float4*>(dst + e) = make_float4(y[e], y[e + 1], y[e + 2], y[e + 3]);
      } else {
        float* dst = sQK + ((size_t)kind * T + t) * KS;
#pragma unroll
        for (int e = 0; e < VEC; ++e) dst[stage_pos<K>(e0 + e)] = y[e];
      }
    } else {
      const int gi = task - n_conv;        // (g, t, e0) with e0 fastest
      const int g = gi / (NQ * T);
      const int r = gi - g * NQ * T;
      const int t = r / NQ;
      const int e0 = (r - t * NQ) * VEC;
      Item itg = base;
      itg.hv = h * G + g;
      itg.vt = 0;
      const GlobalSrc<Act, K, BV> src{p, itg};
      const float braw = e0 == 0 ? load_b<Act>(p, itg, t) : 0.0f;  // issued before the gate math
      const float negA = p.gate_mode != 0 ? 0.0f : -expf(__ldg(p.A_log + itg.hv));
      float al[VEC];
      gate_task<Act>(src, p.gate_mode, negA, t, e0, al);
      float* dst = sA + ((size_t)g * T + t) * KS;
#pragma unroll
      for (int e = 0; e < VEC; ++e) dst[stage_pos<K>(e0 + e)] = al[e];
      if (e0 == 0) sB[(size_t)g * round4(T) + t] = sigmoid_f(braw);
    }
  }
  __syncthreads();  // every conv_state read of the group is done; staging complete
  for (int r = warp; r < 2 * T; r += kPrepThreads / 32) l2norm_warp<K>(sQK + (size_t)r * KS, r < T, lane);
  // roll the group's conv_state to the staged windows
  for (int cv = tid; cv < NCV; cv += kPrepThreads) {
    const int kind = cv < NQ ? 0 : (cv < 2 * NQ ? 1 : 2);
    const int g = kind == 2 ? (cv - 2 * NQ) / NVV : 0;
    const int e0 = kind == 2 ? (cv - 2 * NQ - g * NVV) * VEC : (cv - kind * NQ) * VEC;
    Item itg = base;
    itg.hv = h * G + g;
    itg.vt = 0;
    const int c = block_channel<K, BV>(p, itg, kind) + e0;
    char* cp = reinterpret_cast<char*>(static_cast<Act*>(p.conv_state) +
                                       ((size_t)base.cs_row * p.dim + c) * (kConvW - 1));
#pragma unroll
    for (int m = 0; m < 3; ++m) st_16(cp + 16 * m, stash[3 * cv + m]);
  }
  __syncthreads();  // norms done
  // every item's stage, at its home: item (g, vt) of the group
  const int SF4 = stage_floats(T, K, BV) / 4;
  const int nitems = G * p.nvt;
  const int qk4 = 2 * T * KS / 4, a4 = T * KS / 4, v4 = T * BV / 4;
  for (int i = tid; i < nitems * SF4; i += kPrepThreads) {
    const int j = i / SF4;
    const int s4 = i - j * SF4;
    const int g = j / p.nvt;
    const int vt = j - g * p.nvt;
    const float* src;
    if (s4 < qk4) {
      src = sQK + 4 * s4;
    } else if (s4 < qk4 + a4) {
      src = sA + (size_t)g * T * KS + 4 * (s4 - qk4);
    } else if (s4 < qk4 + a4 + v4) {
      const int idx = 4 * (s4 - qk4 - a4);
      const int t = idx / BV;
      src = sV + ((size_t)g * T + t) * V + vt * BV + (idx - t * BV);
    } else {
      src = sB + (size_t)g * round4(T) + 4 * (s4 - qk4 - a4 - v4);
    }
    Item itg = base;
    itg.hv = h * G + g;
    itg.vt = vt;
    float* home = stage_home<K, BV>(p, itg);
    const int sidx = 4 * s4;
    *reinterpret_cast<float4*>(home + (size_t)(sidx / BV) * V + (sidx % BV)) =
        *reinterpret_cast<const float4*>(src);
  }
}

// ---------------------------------------------------------------------------
// persistent and warp-specialised: producer warps stage the next item while
// consumer warps run the recurrence of the current one
// ---------------------------------------------------------------------------
// Each CTA walks the items blockIdx.x, blockIdx.x + gridDim.x, ...  Every
// input an item needs is requested one item ahead: its raw inputs (token
// rows, conv_state / conv_w / gate rows) by 1-D bulk copies into one of two
// raw buffers, its beta logits and A_log by plain loads into registers, its
// state tile by a 2-D TMA load into the single tile buffer once the consumers
// hold the previous tile in registers.  The producer warps then run the
// producer arithmetic from shared memory into one of two stages while the
// consumer warps stream the previous item's snapshots out, so per SM the
// snapshot writes of one item overlap all the latency of the next.
__host__ __device__ constexpr int pipe_producer_warps(int cw) { return cw; }
__host__ __device__ constexpr int pipe_threads(int cw) { return (cw + pipe_producer_warps(cw)) * 32; }
__host__ __device__ constexpr int pipe_min_blocks(int cw) { return cw >= 8 ? 1 : 2; }
constexpr int kPipeStages = 2;       // stages and raw buffers (double-buffered)
constexpr int kPipeProducerBar = 1;  // named barrier of the producer warps
constexpr int kPipeConsumerBar = 2;  // named barrier of the consumer warps
constexpr int kPipeExt = 20;         // floats per item of loaded-ahead scalars: b[0..15], -exp(A_log)
constexpr int kPipeExtNegA = 16;

struct PipeBars {
  uint64_t tile_full;                  // the item's state tile landed (1 arrival + tx)
  uint64_t raw_full[kPipeStages];      // the item's raw inputs landed (1 arrival + tx)
  uint64_t stage_full[kPipeStages];    // producers staged the item (1 arrival)
  uint64_t stage_empty[kPipeStages];   // consumers done with the stage (one arrival per warp)
  int abort_flag;                      // set by a warp that gave up a bounded wait
  int last_arrival;                    // q/k counter result, broadcast to the producers
};

// dynamic shared memory: header, tile, stages, staged conv windows, raw
// buffers, loaded-ahead scalars
__host__ __device__ constexpr size_t pipe_smem_bytes(int T, int K, int BV, int ab) {
  return kSmemHeader + sizeof(float) * ((size_t)K * BV + kPipeStages * (size_t)stage_floats(T, K, BV)) +
         round16(roll_stash_bytes(K, BV, ab)) + kPipeStages * round16(raw_bytes(T, K, BV, ab)) +
         sizeof(float) * kPipeStages * kPipeExt;
}

// Bounded wait that also gives up when another warp of the CTA gave up.
__device__ __forceinline__ bool pipe_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}

// Named barrier over `count` threads that also ORs a predicate across them:
// every participating thread learns whether any of them failed.
template <int ID, int COUNT>
__device__ __forceinline__ bool group_sync_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "n"(ID), "n"(COUNT)
      : "memory");
  return r != 0;
}

template <int ID, int COUNT>
__device__ __forceinline__ void group_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(COUNT) : "memory");
}

// First item at or after `item`, stepping by `stride`, that is not a padding
// sequence (num_items when none is left).  Producers and consumers walk the
// same items, so their mbarrier phases stay in step.
__device__ __forceinline__ long long next_live_item(const Params& p, long long item, long long stride) {
  while (item < p.num_items && decode_item(p, item).skip) item += stride;
  return item;
}

template <typename Act, int K, int BV>
__device__ __forceinline__ uint32_t raw_tx_bytes(const Params& p) {
  constexpr int AB = sizeof(Act);
  return static_cast<uint32_t>(AB * (p.T * (2 * K + BV) + (2 * K + BV) * 7 + p.T * K) +
                               (p.gate_mode == 0 ? 4 * K : 0));
}

// 1-D bulk copies of one item's raw inputs into `raw` (SmemSrc layout):
// copies first, first + step, ... of the 4T + 6 (+1 with the softplus gate).
// The caller posts raw_tx_bytes on `bar` once per item.  Issuing a bulk copy
// holds the issuing thread for a while, so the producer warps share them.
template <typename Act, int K, int BV>
__device__ __forceinline__ void issue_raw(const Params& p, const Item& it, unsigned char* raw,
                                          uint64_t* bar, int first, int step) {
  constexpr int AB = sizeof(Act);
  const int T = p.T;
  const SmemSrc<Act, K, BV> L{raw, T};
  const int ncopy = 4 * T + 6 + (p.gate_mode == 0 ? 1 : 0);
  for (int c = first; c < ncopy; c += step) {
    const char* src;
    unsigned char* dst;
    uint32_t bytes;
    if (c < 3 * T) {  // token rows of the q, k and v blocks
      const int t = c / 3, kind = c - 3 * t;
      src = static_cast<const char*>(p.mixed_qkv) +
            (((size_t)it.n * T + t) * p.dim + block_channel<K, BV>(p, it, kind)) * AB;
      dst = raw + L.off_x(kind, t);
      bytes = (kind == 2 ? BV : K) * AB;
    } else if (c < 3 * T + 6) {  // conv_state and conv_w blocks
      const int q = c - 3 * T;
      const int kind = q % 3;
      const int ch = block_channel<K, BV>(p, it, kind);
      const int nch = kind == 2 ? BV : K;
      if (q < 3) {
        src = static_cast<const char*>(p.conv_state) + ((size_t)it.cs_row * p.dim + ch) * 3 * AB;
        dst = raw + L.base_cs() + (size_t)L.blk(kind) * 3 * AB;
        bytes = nch * 3 * AB;
      } else {
        src = static_cast<const char*>(p.conv_w) + (size_t)ch * 4 * AB;
        dst = raw + L.base_w() + (size_t)L.blk(kind) * 4 * AB;
        bytes = nch * 4 * AB;
      }
    } else if (c < 4 * T + 6) {  // gate rows
      const int t = c - 3 * T - 6;
      src = static_cast<const char*>(p.a) + ((((size_t)it.n * T + t) * p.HV + it.hv) * K) * AB;
      dst = raw + L.base_a() + (size_t)t * K * AB;
      bytes = K * AB;
    } else {  // dt_bias row (softplus gate)
      src = reinterpret_cast<const char*>(p.dt_bias + (size_t)it.hv * K);
      dst = raw + L.base_dt();
      bytes = K * 4;
    }
    bulk_load(dst, src, bytes, bar);
  }
}

// Raw bits of the scalars an item's gate tasks need, loaded by one lane each
// (lane t < T: b[n, t, hv]; lane kPipeExtNegA: A_log[hv]); to_ext converts
// them once they are needed, so the loads stay in flight meanwhile.
template <typename Act>
__device__ __forceinline__ uint32_t load_ext_bits(const Params& p, const Item& it, int lane) {
  if (lane < p.T) {
    const Act* bp = static_cast<const Act*>(p.b) + ((size_t)it.n * p.T + lane) * p.HV + it.hv;
    if constexpr (sizeof(Act) == 4) return __float_as_uint(__ldg(reinterpret_cast<const float*>(bp)));
    else return static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(bp)));
  }
  if (lane == kPipeExtNegA && p.gate_mode == 0) return __float_as_uint(__ldg(p.A_log + it.hv));
  return 0u;
}
template <typename Act>
__device__ __forceinline__ void store_ext(const Params& p, uint32_t bits, float* ext, int lane) {
  if (lane < p.T) ext[lane] = ActT<Act>::to_f(bits);
  else if (lane == kPipeExtNegA) ext[lane] = p.gate_mode == 0 ? -expf(__uint_as_float(bits)) : 0.0f;
}

template <typename Act, int K, int CW>
__global__ void __launch_bounds__(pipe_threads(CW), pipe_min_blocks(CW))
    kda_pipe_kernel(const __grid_constant__ CUtensorMap tmap_s0, const Params p) {
  constexpr int BV = CW * warp_cols(K);
  constexpr int R = rows_per_thread(K);
  constexpr int KS = stage_ks(K);
  constexpr int PW = pipe_producer_warps(CW);
  constexpr int NP = PW * 32;
  constexpr int NC = CW * 32;
  constexpr int AB = sizeof(Act);
  constexpr int NQV = 2 * K / ActT<Act>::VEC;  // q/k channel vectors
  constexpr int NCV = NQV + BV / ActT<Act>::VEC;
  static_assert(K % 32 == 0 && K <= 128, "K must be 32, 64 or 128");

  extern __shared__ __align__(128) unsigned char smem[];
  PipeBars* bars = reinterpret_cast<PipeBars*>(smem);
  volatile int* abort_flag = &bars->abort_flag;
  float* sbuf = tile_base(smem);
  const int T = p.T;
  const int sf = stage_floats(T, K, BV);
  float* stage0 = sbuf + K * BV;
  uint4* stash = reinterpret_cast<uint4*>(stage0 + kPipeStages * sf);
  const size_t raw_stride = round16(raw_bytes(T, K, BV, AB));
  unsigned char* raw0 = reinterpret_cast<unsigned char*>(stash) + round16(roll_stash_bytes(K, BV, AB));
  float* ext0 = reinterpret_cast<float*>(raw0 + kPipeStages * raw_stride);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long stride = gridDim.x;
  // launched as a programmatic dependent of the stream's previous kernel:
  // nothing global is touched before it has completed.  Then a programmatic
  // dependent of this grid (the q/k roll kernel, or the next call) may be
  // scheduled once every CTA has got here; it waits for this one's end.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const long long first = next_live_item(p, blockIdx.x, stride);
  if (threadIdx.x == 0) {  // report out-of-range slots of this CTA's items
    for (long long i = blockIdx.x; i < p.num_items; i += stride) {
      const Item q = decode_item(p, i);
      if (q.bad && q.hv == 0 && q.vt == 0) atomicOr(p.status, kStatusBadIndex);
    }
  }
  if (first >= p.num_items) return;

  if (threadIdx.x == 0) {
    mbar_init(&bars->tile_full, 1);
    for (int s = 0; s < kPipeStages; ++s) {
      mbar_init(&bars->raw_full[s], 1);
      mbar_init(&bars->stage_full[s], 1);
      mbar_init(&bars->stage_empty[s], CW);
    }
    bars->abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmap_s0);
    const Item it = decode_item(p, first);
    mbar_arrive_expect_tx(&bars->tile_full, K * BV * sizeof(float));
    tma_load_tile<K, BV>(sbuf, &tmap_s0, it.vt, it.s_unit, &bars->tile_full, l2_policy_evict_first());
  }
  __syncthreads();

  if (warp >= CW) {
    // ------------------------------ producers ------------------------------
    const int ptid = threadIdx.x - NC;
    const int pwarp = warp - CW;
    const int expected = p.G * p.nvt;
    long long item = first;
    int raws = 0;  // raw-input copies issued
    if (pwarp == 0) {  // the first item's inputs: raw buffer 0, scalars now
      const Item it = decode_item(p, item);
      if (lane == 0) mbar_arrive_expect_tx(&bars->raw_full[0], raw_tx_bytes<Act, K, BV>(p));
      issue_raw<Act, K, BV>(p, it, raw0, &bars->raw_full[0], lane, 32);
      store_ext<Act>(p, load_ext_bits<Act>(p, it, lane), ext0, lane);
    }
    raws = 1;
    bool failed = false;
    for (int j = 0; item < p.num_items; ++j) {
      const int s = j % kPipeStages;  // stage, raw buffer and scalar slot of this item
      float* sQ = stage0 + s * sf;
      float* sK = sQ + T * KS;
      float* sA = sK + T * KS;
      float* sV = sA + T * KS;
      float* sB = sV + T * BV;
      const Item it = decode_item(p, item);
      const long long next = next_live_item(p, item + stride, stride);
      // this item's raw inputs, and its stage free (the consumers are done
      // with item j - 2)
      // order this thread's reads of the other raw buffer (item j - 1) before
      // the bulk copies that refill it below
      fence_proxy_async_smem();
      bool ok = pipe_wait(&bars->raw_full[s], (j / kPipeStages) & 1, abort_flag);
      if (ok && j >= kPipeStages)
        ok = pipe_wait(&bars->stage_empty[s], ((j / kPipeStages) - 1) & 1, abort_flag);
      if (group_sync_or<kPipeProducerBar, NP>(!ok)) { failed = true; break; }
      // request the next item's inputs: its raw buffer was last read by item
      // j - 1, whose tasks ended before the previous iteration's last barrier
      // (lane 0 of every producer warp issues its share of the copies)
      uint32_t ext_bits = 0;
      if (next < p.num_items) {
        const Item nx = decode_item(p, next);
        if (lane == 0) {
          if (pwarp == 0) mbar_arrive_expect_tx(&bars->raw_full[s ^ 1], raw_tx_bytes<Act, K, BV>(p));
          issue_raw<Act, K, BV>(p, nx, raw0 + (s ^ 1) * raw_stride, &bars->raw_full[s ^ 1], pwarp, PW);
        }
        if (pwarp == PW - 1) ext_bits = load_ext_bits<Act>(p, nx, lane);
      }
      if (next < p.num_items) ++raws;
      const SmemSrc<Act, K, BV> src{raw0 + s * raw_stride, T};
      const float* ext = ext0 + s * kPipeExt;
      produce_tasks<Act, K, BV>(src, p, it, sQ, sK, sA, sV, sB, stash, ptid, NP, ext, ext + kPipeExtNegA);
      group_sync<kPipeProducerBar, NP>();  // every conv_state read of the item is done
      for (int r = pwarp; r < 2 * T; r += PW) l2norm_warp<K>(r < T ? sQ + r * KS : sK + (r - T) * KS, r < T, lane);
      roll_staged<Act, K, BV>(p, it, stash, NQV, NCV, ptid, NP);  // v: owned by this item
      if (expected == 1) {
        roll_staged<Act, K, BV>(p, it, stash, 0, NQV, ptid, NP);  // the only reader of its q/k
      } else if (!p.qk_roll_kernel) {
        // q/k shared by several items: the last one to arrive on the group's
        // counter resets it and rolls (no CTA ever waits on another)
        if (ptid == 0) {
          int* cnt = p.counters + (size_t)it.n * p.H + it.h;
          __threadfence();  // this item's conv_state reads come first
          const int last = atomicAdd(cnt, 1) == expected - 1;
          if (last) {
            atomicExch(cnt, 0);
            __threadfence();  // every other item's reads come before the stores below
          }
          bars->last_arrival = last;
        }
        group_sync<kPipeProducerBar, NP>();
        if (bars->last_arrival) roll_staged<Act, K, BV>(p, it, stash, 0, NQV, ptid, NP);
      }
      if (pwarp == PW - 1 && next < p.num_items) store_ext<Act>(p, ext_bits, ext0 + (s ^ 1) * kPipeExt, lane);
      group_sync<kPipeProducerBar, NP>();  // stage complete; stash free; next scalars visible
      if (ptid == 0) mbar_arrive(&bars->stage_full[s]);
      item = next;
    }
    if (failed && ptid == 0) {
      // report, then let the newest raw copy in flight land before leaving
      *abort_flag = 1;
      atomicOr(p.status, kStatusTmaTimeout);
      const int r = raws - 1;
      mbar_wait_bounded(&bars->raw_full[r % kPipeStages], (r / kPipeStages) & 1, kWaitLimitNs);
    }
  } else {
    // ------------------------------ consumers ------------------------------
    long long item = first;
    int tiles = 1;  // state tile loads issued (the first one above)
    bool failed = false;
    for (int j = 0; item < p.num_items; ++j) {
      const int s = j % kPipeStages;
      const long long next = next_live_item(p, item + stride, stride);
      const Item it = decode_item(p, item);
      bool ok = pipe_wait(&bars->tile_full, j & 1, abort_flag);
      float4 sreg[R];
      if (ok) load_tile<K, BV>(sbuf, sreg, warp, lane);
      fence_proxy_async_smem();  // these tile reads come before the next tile's TMA writes
      if (group_sync_or<kPipeConsumerBar, NC>(!ok)) { failed = true; break; }
      // every consumer holds its part of the tile: load the next item's
      if (threadIdx.x == 0 && next < p.num_items) {
        const Item nx = decode_item(p, next);
        mbar_arrive_expect_tx(&bars->tile_full, K * BV * sizeof(float));
        tma_load_tile<K, BV>(sbuf, &tmap_s0, nx.vt, nx.s_unit, &bars->tile_full, l2_policy_evict_first());
      }
      if (next < p.num_items) ++tiles;
      ok = pipe_wait(&bars->stage_full[s], (j / kPipeStages) & 1, abort_flag);
      if (group_sync_or<kPipeConsumerBar, NC>(!ok)) { failed = true; break; }
      const float* st = stage0 + s * sf;
      consume<Act, K, BV>(p, it, st, st + T * KS, st + 2 * T * KS, st + 3 * T * KS,
                          st + 3 * T * KS + T * BV, sreg, warp, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->stage_empty[s]);
      item = next;
    }
    if (failed && threadIdx.x == 0) {
      // report, then let the newest tile load in flight land before leaving
      *abort_flag = 1;
      atomicOr(p.status, kStatusTmaTimeout);
      mbar_wait_bounded(&bars->tile_full, (tiles - 1) & 1, kWaitLimitNs);
    }
  }
}

}  // namespace kda
