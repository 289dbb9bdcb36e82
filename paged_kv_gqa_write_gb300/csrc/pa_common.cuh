// pa_common.cuh -- device helpers shared by the paged-attention kernels
// (sm_103a): mbarriers with bounded waits, TMA tile loads, named barriers,
// bf16 unpacking and the launch-parameter structs.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pagedattn.h"

namespace pa {

constexpr int kHeadDim = 128;
constexpr int kPage = 128;
// A bounded wait gives up after this much wall-clock time (ns), or after
// kMaxPolls polls, whichever comes first.  Legitimate waits (one page load)
// last microseconds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kMaxPolls = 1u << 30;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
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

// Waits for the phase with the given parity to complete; returns false (after
// recording PA_STATUS_TIMEOUT) if it does not within the limits above.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1; i < kMaxPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 1023u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) break;
  }
  if (status) atomicOr(status, PA_STATUS_TIMEOUT);
  return false;
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 2-D tiled bulk tensor load global -> shared, completing on `bar`.
// x is the inner (contiguous) coordinate in elements; it must be a multiple of
// 8 for 16-bit data so that the copy starts on a 16-byte boundary.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensor_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- barriers
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- numerics
// Two bf16 in one 32-bit word -> two floats (exact).
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ float4 lds128f(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

// ---------------------------------------------------------------- params
struct DecodeParams {
  const __nv_bfloat16* q;       // [B, Hq, D]
  const int32_t* block_table;   // [B, max_pages]
  const int32_t* context_lens;  // [B]
  void* out;                    // [B, Hq, D]
  float* part_o;                // [B, Hq, S, D] (S > 1)
  float* part_lse;              // [B, Hq, S]
  int32_t* status;
  float scale_log2;             // scale * log2(e)
  int32_t B, Hq, Hkv, G, NG;    // NG head groups of GC heads per KV head
  int32_t num_pages, max_pages;
  int32_t pps;                  // pages per split
  int32_t S;                    // splits
  int32_t num_items;            // S * B * Hkv * NG
  int32_t out_f32;
};

struct CombineParams {
  const float* part_o;
  const float* part_lse;
  void* out;
  int32_t rows;  // B * Hq
  int32_t S;
  int32_t out_f32;
};

struct KvWriteParams {
  const uint4* k_new;
  const uint4* v_new;
  uint4* k_cache;
  uint4* v_cache;
  const int32_t* block_table;
  const int32_t* context_lens;
  const int32_t* chunk_lens;  // may be null
  int32_t* status;
  int32_t B, T, Hkv, num_pages, max_pages;
};

struct PrefillParams {
  const __nv_bfloat16* q;       // [T, Hq, D]
  const int32_t* block_table;
  const int32_t* context_lens;
  const int32_t* chunk_lens;
  void* out;                    // [T, Hq, D]
  int32_t* status;
  float scale_log2;
  int32_t B, T, Hq, Hkv, G;
  int32_t num_pages, max_pages;
  int32_t out_f32;
};

}  // namespace pa
