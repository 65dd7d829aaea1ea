// kda_device.cuh -- low-level device helpers for the sm_103a verify-decode
// kernels: inline PTX for mbarriers and TMA tile loads, L2 cache policies,
// 16-byte global accesses and activation-type traits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

// ---------------------------------------------------------------------------
// shared-memory addressing, mbarrier, TMA
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Make the initialised barrier visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of `bar` to complete, giving up after ~limit_ns.
// Returns false on time-out (the caller reports it and never spins forever).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
  }
}

// Thread-block cluster barrier, split in its two halves.  Every thread of
// every CTA of the cluster arrives once (release: its earlier memory accesses
// are ordered before the arrival) and later waits (acquire).  The wait ends
// once all threads of the cluster have arrived; the hardware schedules the
// CTAs of a cluster together, so a CTA that arrives before any wait of its
// own never leaves another waiting forever.
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// L2 policy: lines read once (the persistent state tile) go first.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 2-D TMA tile load, global -> this CTA's shared memory, completion counted
// in bytes on `bar`.  x is the innermost (contiguous) coordinate.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 1-D bulk copy (TMA engine), global -> this CTA's shared memory, completion
// counted in bytes on `bar`.  Both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// L2 prefetch of a 2-D TMA tile (no shared memory, no completion to wait on).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

// L2 prefetch of a contiguous range (16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)),
               "r"(bytes)
               : "memory");
}

// ---------------------------------------------------------------------------
// 16-byte global accesses
// ---------------------------------------------------------------------------

// Read-only for the whole kernel: non-coherent path.
__device__ __forceinline__ uint4 ld_ro_16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
// Data that this kernel also writes (conv_state): coherent L2 path.
__device__ __forceinline__ uint4 ld_rw_16(const void* p) {
  return __ldcg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st_16(void* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// Streaming (evict-first) 16-byte store of a state snapshot.
__device__ __forceinline__ void st_stream_f4(float* p, float4 v) {
  __stcs(reinterpret_cast<float4*>(p), v);
}

// ---------------------------------------------------------------------------
// activation types: raw bits, unpack to fp32, 16-byte packing
// ---------------------------------------------------------------------------

template <typename Act>
struct ActT;

template <>
struct ActT<float> {
  using Raw = uint32_t;
  static constexpr int VEC = 4;  // elements per 16 bytes
  __device__ static __forceinline__ float to_f(Raw r) { return __uint_as_float(r); }
  __device__ static __forceinline__ void unpack(const uint4& u, Raw* r) {
    r[0] = u.x; r[1] = u.y; r[2] = u.z; r[3] = u.w;
  }
  // pack 4 raw values starting at r into one 16-byte word
  __device__ static __forceinline__ uint4 pack(const Raw* r) {
    return make_uint4(r[0], r[1], r[2], r[3]);
  }
  __device__ static __forceinline__ void store4(void* p, float4 v) {
    *reinterpret_cast<float4*>(p) = v;
  }
};

template <>
struct ActT<__nv_bfloat16> {
  using Raw = uint32_t;  // 16 significant bits, kept in a 32-bit register
  static constexpr int VEC = 8;
  __device__ static __forceinline__ float to_f(Raw r) { return __uint_as_float(r << 16); }
  __device__ static __forceinline__ void unpack(const uint4& u, Raw* r) {
    r[0] = u.x & 0xffffu; r[1] = u.x >> 16;
    r[2] = u.y & 0xffffu; r[3] = u.y >> 16;
    r[4] = u.z & 0xffffu; r[5] = u.z >> 16;
    r[6] = u.w & 0xffffu; r[7] = u.w >> 16;
  }
  __device__ static __forceinline__ uint4 pack(const Raw* r) {
    return make_uint4(r[0] | (r[1] << 16), r[2] | (r[3] << 16), r[4] | (r[5] << 16),
                      r[6] | (r[7] << 16));
  }
  // four fp32 results -> four bf16 (round to nearest even), one 8-byte store
  __device__ static __forceinline__ void store4(void* p, float4 v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 w;
    w.x = *reinterpret_cast<uint32_t*>(&lo);
    w.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p) = w;
  }
};

// ---------------------------------------------------------------------------
// scalar math shared by every variant (same formula => bit-identical results)
// ---------------------------------------------------------------------------

// The producer's activations sit on the critical path of every item, so they
// use the hardware exponential / logarithm (__expf, __logf) and the
// approximate divide: relative errors of a few 1e-7 up to ~1e-5 (exponent
// magnitudes up to ~90), far inside the verify tolerance (2e-3), and
// measured 1-4 % faster on whole calls than the IEEE-rounded forms.
// Overflow is harmless: 1 + __expf(..) = inf makes the quotient 0.

__device__ __forceinline__ float silu_f(float y) { return __fdividef(y, 1.0f + __expf(-y)); }

__device__ __forceinline__ float sigmoid_f(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// softplus with threshold 20 as a real branch: the exponential is never
// evaluated where it could overflow, so no 0 * inf can appear.  Below the
// threshold log(1 + e), e = exp(x): where e < 1e-3 the first two terms of the
// series e - e^2/2 + e^3/3 - ... (relative truncation error < e^2/3 < 4e-7),
// which keeps the tiny values that log(1 + e) rounds away; __logf elsewhere.
__device__ __forceinline__ float softplus_f(float x) {
  if (x > 20.0f) return x;
  const float e = __expf(x);
  return e < 1e-3f ? __fmaf_rn(-0.5f * e, e, e) : __logf(1.0f + e);
}

// alpha = exp(g) of the gate (g <= 0)
__device__ __forceinline__ float decay_f(float g) { return __expf(g); }

}  // namespace kda
