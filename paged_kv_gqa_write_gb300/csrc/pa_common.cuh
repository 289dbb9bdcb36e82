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
// Longest a waiting thread sleeps per poll (it wakes earlier when the phase completes).
constexpr uint32_t kSleepHintNs = 20000;

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

// This thread's generic-proxy global writes, ordered before later async-proxy
// (TMA) accesses that a barrier orders after them.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
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

// As above, but the thread may sleep up to `hint_ns` waiting for the phase
// instead of returning at once, so a waiting warp does not take issue slots
// from the other warps of its SM sub-partition.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for the phase with the given parity to complete; returns false (after
// recording PA_STATUS_TIMEOUT) if it does not within limit_ns of wall-clock
// time or kMaxPolls polls.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, int32_t* status,
                                              uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1; i < kMaxPolls; ++i) {
    if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if ((i & 15u) == 0 && global_timer_ns() - t0 > limit_ns) break;
  }
  if (status) atomicOr(status, PA_STATUS_TIMEOUT);
  return false;
}

// The kernels' wait: the limit above (kWaitLimitNs).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* status) {
  return mbar_wait_for(bar, parity, status, kWaitLimitNs);
}

// ---------------------------------------------------------------- clusters
// Cluster-scope forms for a CTA pair: a wait whose phase other CTAs of the
// cluster complete (remote arrivals, multicast commits, paired TMA), and the
// arrival on a barrier of another CTA.
__device__ __forceinline__ bool mbar_try_wait_sleep_cl(uint64_t* bar, uint32_t parity,
                                                       uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cl_for(uint64_t* bar, uint32_t parity, int32_t* status,
                                                 uint64_t limit_ns) {
  if (mbar_try_wait_sleep_cl(bar, parity, 0)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1; i < kMaxPolls; ++i) {
    if (mbar_try_wait_sleep_cl(bar, parity, kSleepHintNs)) return true;
    if ((i & 15u) == 0 && global_timer_ns() - t0 > limit_ns) break;
  }
  if (status) atomicOr(status, PA_STATUS_TIMEOUT);
  return false;
}

__device__ __forceinline__ bool mbar_wait_cl(uint64_t* bar, uint32_t parity, int32_t* status) {
  return mbar_wait_cl_for(bar, parity, status, kWaitLimitNs);
}

__device__ __forceinline__ bool mbar_wait_warp_cl(uint64_t* bar, uint32_t parity,
                                                  int32_t* status) {
  const bool ok = mbar_wait_cl(bar, parity, status);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// All threads of every CTA of the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared::cluster address of this CTA's shared variable at `saddr` in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// Hand this thread's shared::cta writes (and those it has synchronised with,
// e.g. its warp's after __syncwarp) to a consumer in another CTA: a release
// fence at cluster scope restricted to shared::cta accesses, then a relaxed
// arrival on the barrier at shared::cluster address `caddr`.  The restricted
// fence does not wait for global memory, so it costs about as much as a
// local arrival; the consumer's cluster-scope acquire pairs with it.
__device__ __forceinline__ void mbar_arrive_cluster_smem(uint32_t caddr) {
  asm volatile("fence.sync_restrict::shared::cta.release.cluster;" ::: "memory");
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr)
               : "memory");
}

// Arrive (release at cluster scope) on the barrier at shared::cluster address `caddr`.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t caddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr)
               : "memory");
}

// Warp-uniform variant: every lane waits and all lanes agree on the outcome,
// so a timeout never leaves a warp diverged before a .sync.aligned operation.
__device__ __forceinline__ bool mbar_wait_warp_for(uint64_t* bar, uint32_t parity,
                                                   int32_t* status, uint64_t limit_ns) {
  const bool ok = mbar_wait_for(bar, parity, status, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, int32_t* status) {
  return mbar_wait_warp_for(bar, parity, status, kWaitLimitNs);
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

// 3-D tiled bulk tensor load global -> shared (x innermost, in elements).
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, int32_t z, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)),
      "l"(policy)
      : "memory");
}

// Paired-CTA forms (.cta_group::2): the data lands in this CTA's shared
// memory and the byte count completes on the barrier at shared::cluster
// address `bar_cl`, which may belong to the other CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map, int32_t x,
                                                 int32_t y, uint32_t bar_cl, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".cta_group::2.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cl), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(void* smem_dst, const CUtensorMap* map, int32_t x,
                                                 int32_t y, int32_t z, uint32_t bar_cl,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".cta_group::2.L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar_cl), "l"(policy)
      : "memory");
}

// 3-D tiled bulk tensor store shared -> global (x innermost, in elements),
// tracked by the issuing thread's bulk async-group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* smem_src, int32_t x,
                                             int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(smem_src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// This thread's committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// This thread's committed bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// ---------------------------------------------------------------- tcgen05
// Tensor memory (TMEM) is allocated in columns by one whole warp; the address
// (lane in bits 31..16, column in bits 15..0) is written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_result, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_result)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// CTA-pair (cta_group::2) forms: one warp of each CTA of the pair allocates
// and frees together; the same columns are allocated in both CTAs.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* smem_result, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_result)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Instruction descriptor of tcgen05.mma kind::f16 with BF16 A and B, FP32
// accumulate, an M x N tile; *_mn selects MN-major (transposed) operands.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4)                            // D format: F32
         | (1u << 7)                          // A format: BF16
         | (1u << 10)                         // B format: BF16
         | ((a_mn ? 1u : 0u) << 15)           // A major
         | ((b_mn ? 1u : 0u) << 16)           // B major
         | ((uint32_t)(N >> 3) << 17)         // N / 8
         | ((uint32_t)(M >> 4) << 24);        // M / 16
}

// The same with F16 A and B (the FP8-cache decode: e4m3 values are exact in F16).
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4)                            // D format: F32
         | ((a_mn ? 1u : 0u) << 15)           // A major (A and B format 0: F16)
         | ((b_mn ? 1u : 0u) << 16)           // B major
         | ((uint32_t)(N >> 3) << 17)         // N / 8
         | ((uint32_t)(M >> 4) << 24);        // M / 16
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand whose
// swizzle atoms (8 rows of 128 bytes) start on 1024-byte boundaries.
// lbo / sbo: leading / stride byte offsets of the canonical layout.
__device__ __forceinline__ uint64_t umma_sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;  // layout: 128-byte swizzle
  return d;
}

// D[tmem] (+)= A[smem] * B[smem], issued by one thread.
__device__ __forceinline__ void umma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (+)= A * B across a CTA pair (cta_group::2, M = 256): each CTA supplies
// its 128 rows of A and half of B's N columns from the same shared-memory
// offsets, and holds its 128 rows of D in its own tensor memory.  Issued by
// one thread of the even CTA.
__device__ __forceinline__ void umma_bf16_ss_pair(uint32_t d_tmem, uint64_t a_desc,
                                                  uint64_t b_desc, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same with A from tensor memory: each CTA's 128 lanes at column a_tmem
// hold its rows of A (M x 16 BF16, a pair per 32-bit column).
__device__ __forceinline__ void umma_bf16_ts_pair(uint32_t d_tmem, uint32_t a_tmem,
                                                  uint64_t b_desc, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the barrier at this shared offset in every CTA of `mask`
// when all pair MMAs this thread issued so far are done.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// Arrive (once) on `bar` when every tcgen05 op this thread issued so far is done.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 consecutive 32-bit TMEM columns of this thread's lane -> registers.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
      "%10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, "
      "%27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
      "%10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// ---------------------------------------------------------------- barriers
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Barrier `id` over `nthreads` threads that also ORs a predicate across them.
__device__ __forceinline__ bool named_bar_red_or(bool v, int id, int nthreads) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, %2, %3, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void sts64(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// ---------------------------------------------------------------- numerics
// Two floats -> two F16 (round to nearest even) in one 32-bit word, lo first.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two F16 in one 32-bit word -> two floats (exact).
__device__ __forceinline__ float2 f16x2_to_float2(uint32_t w) {
  float2 f;
  asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "cvt.f32.f16 %0, lo;\n\tcvt.f32.f16 %1, hi;\n\t}"
      : "=f"(f.x), "=f"(f.y)
      : "r"(w));
  return f;
}

// 4 e4m3 codes (bytes 0..3 of w) -> 4 F16 values (exact): two F16 pairs.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// 16 e4m3 codes -> 16 F16 values (exact), as two 16-byte chunks.
__device__ __forceinline__ void e4m3x16_to_f16(uint4 c, uint4& lo, uint4& hi) {
  e4m3x4_to_f16x4(c.x, lo.x, lo.y);
  e4m3x4_to_f16x4(c.y, lo.z, lo.w);
  e4m3x4_to_f16x4(c.z, hi.x, hi.y);
  e4m3x4_to_f16x4(c.w, hi.z, hi.w);
}

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

// ---------------------------------------------------------------- token -> slot
// (used by the kernels that write new tokens into the cache)
// Inclusive prefix sums of max(chunk_lens, 0) into off[0..B), built by the
// whole block.  Returns (in every thread) whether any chunk length was negative.
__device__ __forceinline__ bool block_chunk_offsets(const int32_t* chunk_lens, int B, int32_t* off,
                                    int32_t* scratch /* blockDim.x ints */) {
  const int nt = blockDim.x, tid = threadIdx.x;
  const int per = (B + nt - 1) / nt;
  const int lo = min(B, tid * per), hi = min(B, lo + per);
  int sum = 0, neg = 0;
  for (int i = lo; i < hi; ++i) {
    int c = chunk_lens[i];
    neg |= c < 0;
    sum += c > 0 ? c : 0;
    off[i] = sum;
  }
  // exclusive prefix of the per-thread sums: a scan within each warp, then one
  // over the warp totals (blockDim.x is a multiple of 32, at most 1024)
  const int lane = tid & 31, w = tid >> 5, nw = nt >> 5;
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) scratch[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int v = lane < nw ? scratch[lane] : 0;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += t;
    }
    if (lane < nw) scratch[lane] = x - v;
  }
  __syncthreads();
  const int base = scratch[w] + incl - sum;
  for (int i = lo; i < hi; ++i) off[i] += base;
  return __syncthreads_or(neg) != 0;
}

// Sequence holding packed token `token`: the first s with off[s] > token, or B.
__device__ __forceinline__ int seq_of_token(const int32_t* off, int B, int token) {
  int lo = 0, hi = B;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (off[mid] > token) hi = mid; else lo = mid + 1;
  }
  return lo;
}

// Warp-wide check that sequence s has consistent lengths and that every
// block-table entry it references lies in [0, num_pages).  Returns 0 when
// valid, else a PA_STATUS_* bit.
__device__ __forceinline__ int warp_check_sequence(const int32_t* block_table, int s, int ctx, int n,
                                   int num_pages, int max_pages) {
  if (ctx < 0 || n < 0 || n > ctx || ctx > max_pages * kPage) return PA_STATUS_BAD_LENGTH;
  const int used = (ctx + kPage - 1) / kPage;
  const int lane = threadIdx.x & 31;
  const int32_t* row = block_table + (int64_t)s * max_pages;
  bool bad = false;
  for (int i = lane; i < used; i += 32) {
    int p = row[i];
    bad |= (p < 0 || p >= num_pages);
  }
  return __any_sync(0xffffffffu, bad) ? PA_STATUS_BAD_PAGE : 0;
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
  int32_t B, Hq, Hkv, G;
  int32_t L;                    // new tokens (queries) per sequence
  int32_t NT, Lg;               // token groups per KV head, tokens per group
  const float* k_scale;         // FP8 cache: [Hkv] per-head K and V scales (else null)
  const float* v_scale;
  int32_t num_pages, max_pages;
  int32_t pps;                  // pages per split
  int32_t S;                    // splits
  int32_t num_items;            // S * B * Hkv * NG (fixed splits)
  int32_t out_f32;
  int32_t balanced;             // page-balanced schedule instead of fixed splits
  int32_t grid;                 // CTAs of the page-balanced schedule (groups x Hkv*NG)
  float* bal_o;                 // [2 * grid][16][D] partial records of cut sequences
  float* bal_lse;               // [2 * grid][16]
};

// Decode with L new tokens per sequence (multi-token decode; L = 1 is the
// plain decode): token t of sequence s sits at position context_lens[s] - L + t
// and sees keys 0 .. that position.  A work item serves one KV head and a
// group of Lg consecutive tokens: its MMA columns are (token, query head)
// pairs, token-major, so every K/V page it loads serves all of them.  The
// item reads the sequence's pages up to context_lens[s] (its last token's
// keys); column c masks keys at or past context_lens[s] - (L - 1 - t(c)).
// A sequence with 0 < context_lens[s] < L is invalid (-1 here).
__device__ __forceinline__ int seq_ctx(const int32_t* context_lens, int s, int L) {
  const int c = __ldg(context_lens + s);
  return (L > 1 && c > 0 && c < L) ? -1 : c;
}

// ---------------------------------------------------------------- prologue arithmetic
// Shared by the prologue kernel and the decode kernel's in-kernel prologue, so
// that both produce the same bits.

// cos and sin of a NeoX pair's angle at position pos: frequency f radians per
// position, or (th + tl) turns per position as an unevaluated float pair.
// `fast`: pos * th stays below 2^22 turns (and pos below 2^24), so the whole
// turns drop out exactly and the float path keeps full accuracy; otherwise
// the product and its reduction run in double precision.
__device__ __forceinline__ void rope_sincos(int pos, bool fast, float th, float tl, double f,
                                            float& sn, float& cs) {
  if (fast) {
    const float fpos = (float)pos;
    const float hi = fpos * th;
    const float lo = fmaf(fpos, tl, fmaf(fpos, th, -hi));
    sincospif(2.f * ((hi - rintf(hi)) + lo), &sn, &cs);
  } else {
    constexpr double kTwoPiD = 6.283185307179586476925286766559;
    const double a = (double)pos * f;
    sincosf((float)fma(-rint(a * (1.0 / kTwoPiD)), kTwoPiD, a), &sn, &cs);
  }
}

// Whether the float angle path holds at pos (gmax: the largest turn rate).
__device__ __forceinline__ bool rope_fast(int pos, float gmax) {
  return pos < (1 << 24) && (float)pos * gmax < 4194304.f;
}

__device__ __forceinline__ float4 bf16x4_to_float4(uint2 w) {
  const float2 a = bf16x2_to_float2(w.x), b = bf16x2_to_float2(w.y);
  return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ uint2 float4_to_bf16x4(float4 v) {
  return make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
}

// One head's per-head RMSNorm and NeoX rotation, a half-warp per head: lane
// li of the half holds values 4 li .. 4 li + 3 (ra) and 64 + 4 li .. + 3 (rb),
// both members of four pairs (i, i + 64); w*, c4 and s4 are the norm weights
// and the pairs' cos / sin at those indices.  The results, times `post`,
// rounded to bf16: oa (values 4 li ..) and ob (64 + 4 li ..).  Every lane of the
// warp calls it (a 16-lane shuffle reduction).
__device__ __forceinline__ void norm_rope_half(uint2 ra, uint2 rb, float4 wa, float4 wb,
                                               float4 c4, float4 s4, float eps, float post,
                                               float4& oa, float4& ob) {
  const float4 xa = bf16x4_to_float4(ra), xb = bf16x4_to_float4(rb);
  float ss = xa.x * xa.x + xa.y * xa.y + xa.z * xa.z + xa.w * xa.w +
             xb.x * xb.x + xb.y * xb.y + xb.z * xb.z + xb.w * xb.w;
#pragma unroll
  for (int o = 8; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float sc = rsqrtf(ss * (1.f / kHeadDim) + eps) * post;
  const float4 ta = make_float4(xa.x * wa.x, xa.y * wa.y, xa.z * wa.z, xa.w * wa.w);
  const float4 tb = make_float4(xb.x * wb.x, xb.y * wb.y, xb.z * wb.z, xb.w * wb.w);
  // (x_i, x_{i+64}) -> (x_i cos - x_{i+64} sin, x_{i+64} cos + x_i sin), times the scale
  oa = make_float4(fmaf(ta.x, c4.x, -tb.x * s4.x) * sc, fmaf(ta.y, c4.y, -tb.y * s4.y) * sc,
                   fmaf(ta.z, c4.z, -tb.z * s4.z) * sc, fmaf(ta.w, c4.w, -tb.w * s4.w) * sc);
  ob = make_float4(fmaf(tb.x, c4.x, ta.x * s4.x) * sc, fmaf(tb.y, c4.y, ta.y * s4.y) * sc,
                   fmaf(tb.z, c4.z, ta.z * s4.z) * sc, fmaf(tb.w, c4.w, ta.w * s4.w) * sc);
}

// The decode step's prologue run inside the decode kernel (pa_decode_prologue):
// the inputs of pa_qk_norm_rope_write for one new token per sequence.
struct DecodePrologue {
  const __nv_bfloat16* qkv;     // [B, (Hq + 2 Hkv) * D] bf16
  const float* wq;              // [D] Q norm weight
  const float* wk;              // [D] K norm weight
  __nv_bfloat16* k_cache;       // the new token's K and V rows are written here
  __nv_bfloat16* v_cache;
  float eps, q_scale;
  double freq[64];              // the 64 pairs' frequencies, as in PrologueParams
  float turn_hi[64], turn_lo[64];
};

// Q/K RMSNorm -> NeoX RoPE -> KV cache write for the new tokens.
struct PrologueParams {
  const uint2* qkv;             // [T, (Hq + 2 Hkv) * D] bf16, 4 values per uint2
  const float* wq;              // [D] Q norm weight
  const float* wk;              // [D] K norm weight
  uint2* q_out;                 // [T, Hq, D] bf16
  uint2* k_cache;               // [num_pages, 128, Hkv, D] bf16, or e4m3 codes
  uint2* v_cache;
  const float* k_scale;         // [Hkv] FP8 cache scales; null: bf16 cache
  const float* v_scale;
  const int32_t* block_table;
  const int32_t* context_lens;
  const int32_t* chunk_lens;    // may be null (one token per sequence)
  int32_t* status;
  float eps, q_scale;
  int32_t B, T, Hq, Hkv, num_pages, max_pages;
  // RoPE frequencies of the 64 pairs, base^(-2i/D) / scale: in radians per
  // position (double) and in turns per position as an unevaluated float pair
  double freq[64];
  float turn_hi[64], turn_lo[64];
};

// Exact top-k over rows of logits.
struct TopkParams {
  const float* logits;          // [rows] x row_stride floats, the first vocab of each used
  int64_t row_stride;
  float* out_values;            // [rows, k]
  int32_t* out_indices;         // [rows, k]
  unsigned long long* cand;     // [rows, slices, k] candidate keys (workspace)
  int32_t rows, vocab, k;
  int32_t slices, slice_len;    // slices per row of slice_len entries (a multiple of 4)
};

// Merge of the sequences that the page-balanced decode schedule cut between
// CTA groups.
struct BalCombineParams {
  const int32_t* context_lens;
  const float* bal_o;
  const float* bal_lse;
  void* out;
  int32_t B, Hq, G, max_pages;
  int32_t L, NT, Lg;            // new tokens per sequence, token groups, tokens per group
  int32_t grid;                 // CTAs of the decode launch
  int32_t NC;                   // column slots per record (the decode kernel's MMA width)
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
  uint4* k_cache;               // bf16 rows, or e4m3 rows for the FP8 write
  uint4* v_cache;
  const float* k_scale;         // FP8 write: [Hkv] per-head scales (else null)
  const float* v_scale;
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
  const float* k_scale;         // FP8 cache: [Hkv] scales of the K and V codes
  const float* v_scale;
};

}  // namespace pa
