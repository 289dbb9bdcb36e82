// pa_decode.cu -- paged GQA decode attention, flash-decoding split-K.
//
// Computes, for every sequence s and query head g (KV head h = g / G):
//   out[s][g] = softmax(scale * q[s][g] . K_t) V_t over t < context_lens[s],
// with K_t / V_t gathered through the block table ("Qwen3-14B" pypto-lib doc,
// "decode_fwd": paged attention after the KV cache write, vLLM ABI with flat
// [page, token, kv_head, dim] K/V; "Qwen 3" TensorSharp doc, section 11: K/V
// gathered per sequence from the block tables and sequence lengths).
//
// Design (GB300, HBM bound: every K/V byte is read once; about 5 flop/byte):
//  * Persistent grid, one CTA per SM.  A work item is (split j, sequence s,
//    KV head h, head group): a contiguous range of at most `pps` pages.  Items
//    are dealt round-robin (item i -> CTA i mod grid); split boundaries depend
//    only on logical positions, so results never depend on physical pages.
//  * Page tiles stream through a 3-stage ring of 64 KB stages (K and V of one
//    page); a TMA load takes about 3 us under full load, so two stages in
//    flight per SM cover it (a load-only run of this ring reaches the device's
//    copy bandwidth).  Large head groups use two stages, leaving room for
//    their merge buffer.
//  * Stager warp: runs up to two items ahead, converting each item's query
//    heads to FP32 pre-multiplied by scale * log2 e, reading its context
//    length and block-table entries (validity flag + sanitised page ids) into
//    a 2-slot item ring.  TMA warp: one lane issues 2-D TMA loads (two 64-column
//    boxes per tile, 128-byte swizzle, L2 evict-first) of K and V page tiles
//    from those page ids.  Neither the TMA lane nor the consumers wait on
//    global memory.
//  * Eight consumer warps (two per SM sub-partition) share each page; warp w
//    owns tokens 16w..16w+15.  Scores: lane (token, dim half) reads its 64
//    dims of the K row once from shared memory and uses them for all GC query
//    heads (the GQA saving), accumulating with packed FP32 FMAs
//    (fma.rn.f32x2); one shuffle joins the halves.  Softmax: per-warp running
//    max by shuffles, exp2, per-lane partial sums.  P.V: a half-warp per
//    token, each lane owning 8 output dims; tokens past the context are
//    skipped (a select keeps poisoned tail rows out: 0 * NaN would be NaN).
//  * Item end: each warp publishes its (m, l, o) to shared memory and moves on
//    to the next item; one warp (rotating with the item) merges the eight
//    states in a fixed order and writes `out` (one split) or normalised
//    partials (o, lse) for the combine kernel.
#include "pa_launch.cuh"

namespace pa {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kTmaWarp = kConsumerWarps;
constexpr int kStagerWarp = kConsumerWarps + 1;
constexpr int kThreads = kConsumers + 64;
constexpr int kTokPerWarp = kPage / kConsumerWarps;  // 16
constexpr int kBoxBytes = 64 * 2 * kPage;     // 64 dims x 128 tokens of bf16 = 16 KB
constexpr int kStageBytes = 4 * kBoxBytes;    // K lo, K hi, V lo, V hi of a page
constexpr int kListMax = 64;                  // page ids staged per item
constexpr int kSmemLimit = 232448;
constexpr float kLn2 = 0.69314718055994530942f;
// q row: each 64-dim half padded to 68 floats so the two halves a warp reads
// together fall in different shared-memory banks
constexpr int kQHalf = 68;
constexpr int kQRow = 2 * kQHalf;

// Ring stages (64 KB each): three, or two when a large head group's merge
// buffer needs the room.
template <int GC>
constexpr int stages_for() { return GC <= 5 ? 3 : 2; }

template <int GC>
struct Layout {
  static constexpr int kStages = stages_for<GC>();
  static constexpr int PS = 2 * ((GC + 1) & ~1);                 // p row: (p, p) pairs
  static constexpr int q = kStages * kStageBytes;                // q [2][GC][kQRow] f32
  static constexpr int info = q + 2 * GC * kQRow * 4;            // [2][2] int: flag, ctx
  static constexpr int list = info + 16;                         // [2][kListMax] int
  static constexpr int p = list + 2 * kListMax * 4;              // p_s [8][16][PS] f32
  static constexpr int mml = p + kConsumerWarps * kTokPerWarp * PS * 4;  // m,l [8][GC][2]
  static constexpr int mo = (mml + kConsumerWarps * GC * 2 * 4 + 15) & ~15;  // o [8][GC][128]
  static constexpr int bars = mo + kConsumerWarps * GC * kHeadDim * 4;
  static constexpr int kNumBars = 2 * kStages + 4 + 2;
  static constexpr int total = bars + 8 * kNumBars;
  static constexpr int alloc = total + 1024;                     // room to align to 1024 B
};

struct Item {
  int s, h, hg, j, pg0, pg1, ctx;
  bool ok;
};

__device__ __forceinline__ int item_seq(int i, const DecodeParams& p) {
  const int per_seq = p.Hkv * p.NG;
  return (i % (p.B * per_seq)) / per_seq;
}

__device__ __forceinline__ Item decode_item(int i, const DecodeParams& p, int ctx) {
  Item it;
  const int per_seq = p.Hkv * p.NG;
  const int U = p.B * per_seq;
  it.j = i / U;
  const int u = i - it.j * U;
  it.s = u / per_seq;
  const int r = u - it.s * per_seq;
  it.h = r / p.NG;
  it.hg = r - it.h * p.NG;
  it.ctx = ctx;
  it.ok = it.ctx >= 0 && it.ctx <= p.max_pages * kPage;
  const int npg = it.ok ? (it.ctx + kPage - 1) / kPage : 0;
  it.pg0 = it.j * p.pps;
  it.pg1 = min(npg, it.pg0 + p.pps);
  if (it.pg1 < it.pg0) it.pg1 = it.pg0;
  return it;
}

template <int GC>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  using L = Layout<GC>;
  constexpr int kStages = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* empty = full + kStages;
  uint64_t* ifull = empty + kStages;        // item slot staged
  uint64_t* iempty = ifull + 2;             // item slot consumed
  uint64_t* merge_ready = iempty + 2;       // all warps published their state
  uint64_t* merge_free = merge_ready + 1;   // the merging warp has read it
  float* q_ring = reinterpret_cast<float*>(smem + L::q);
  int* info = reinterpret_cast<int*>(smem + L::info);
  int* plist = reinterpret_cast<int*>(smem + L::list);
  float* p_s = reinterpret_cast<float*>(smem + L::p);
  float* m_ml = reinterpret_cast<float*>(smem + L::mml);
  float* m_o = reinterpret_cast<float*>(smem + L::mo);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ifull[i], 32);
      mbar_init(&iempty[i], kConsumerWarps + 1);
    }
    mbar_init(merge_ready, kConsumerWarps);
    mbar_init(merge_free, 1);
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kStagerWarp) {
    // ------------------------------------------------------------ stager warp
    uint32_t n = 0;
    for (int i = blockIdx.x; i < p.num_items; i += gridDim.x, ++n) {
      const int slot = n & 1;
      if (!mbar_wait_warp(&iempty[slot], ((n >> 1) & 1) ^ 1, p.status)) return;
      const Item it = decode_item(i, p, __ldg(p.context_lens + item_seq(i, p)));
      // query heads of the item -> FP32 * scale * log2(e); lane owns 4 dims
      const int head0 = it.h * p.G + it.hg * GC;
      const uint2* qg =
          reinterpret_cast<const uint2*>(p.q + ((int64_t)it.s * p.Hq + head0) * kHeadDim);
      float* qd = q_ring + slot * GC * kQRow + (lane >> 4) * kQHalf + (lane & 15) * 4;
#pragma unroll
      for (int g = 0; g < GC; ++g) {
        const uint2 w = __ldg(qg + g * (kHeadDim / 4) + lane);
        const float2 a = bf16x2_to_float2(w.x), b = bf16x2_to_float2(w.y);
        *reinterpret_cast<float4*>(qd + g * kQRow) =
            make_float4(a.x * p.scale_log2, a.y * p.scale_log2, b.x * p.scale_log2,
                        b.y * p.scale_log2);
      }
      // validity of every page the item reads, and the sanitised page ids
      const int32_t* bt = p.block_table + (int64_t)it.s * p.max_pages;
      bool bad = false;
      for (int pg = it.pg0 + lane; pg < it.pg1; pg += 32) {
        const int pid = __ldg(bt + pg);
        const bool inval = pid < 0 || pid >= p.num_pages;
        bad |= inval;
        if (pg - it.pg0 < kListMax) plist[slot * kListMax + pg - it.pg0] = inval ? 0 : pid;
      }
      bad = __any_sync(0xffffffffu, bad) || !it.ok;
      if (lane == 0) {
        info[2 * slot] = bad ? (it.ok ? 1 : 2) : 0;
        info[2 * slot + 1] = it.ctx;
      }
      mbar_arrive(&ifull[slot]);
    }
    return;
  }

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA warp
    if (lane == 0) {
      prefetch_tensor_map(&tm_k);
      prefetch_tensor_map(&tm_v);
      const uint64_t pol = l2_policy_evict_first();
      int rs = 0;
      uint32_t rph = 0, n = 0;
      for (int i = blockIdx.x; i < p.num_items; i += gridDim.x, ++n) {
        const int slot = n & 1;
        if (!mbar_wait(&ifull[slot], (n >> 1) & 1, p.status)) return;
        const Item it = decode_item(i, p, info[2 * slot + 1]);
        const int32_t* bt = p.block_table + (int64_t)it.s * p.max_pages;
        const int x = it.h * kHeadDim;
        for (int pg = it.pg0; pg < it.pg1; ++pg) {
          int page;
          if (pg - it.pg0 < kListMax) {
            page = plist[slot * kListMax + pg - it.pg0];
          } else {
            page = __ldg(bt + pg);
            if (page < 0 || page >= p.num_pages) page = 0;  // output is zeroed anyway
          }
          const int y = page * kPage;
          if (!mbar_wait(&empty[rs], rph ^ 1, p.status)) return;
          mbar_arrive_expect_tx(&full[rs], kStageBytes);
          uint8_t* dst = smem + rs * kStageBytes;
          tma_load_2d(dst, &tm_k, x, y, &full[rs], pol);
          tma_load_2d(dst + kBoxBytes, &tm_k, x + 64, y, &full[rs], pol);
          tma_load_2d(dst + 2 * kBoxBytes, &tm_v, x, y, &full[rs], pol);
          tma_load_2d(dst + 3 * kBoxBytes, &tm_v, x + 64, y, &full[rs], pol);
          if (++rs == kStages) { rs = 0; rph ^= 1; }
        }
        mbar_arrive(&iempty[slot]);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int tq = lane & 15, dh = lane >> 4;    // scores: token of the warp's slice, dim half
  const int half = lane >> 4, jd = lane & 15;  // P.V: token parity, 8-dim chunk
  const uint32_t p_addr = smem_u32(p_s) + warp * kTokPerWarp * L::PS * 4;
  int rs = 0;
  uint32_t rph = 0, n = 0;

  for (int i = blockIdx.x; i < p.num_items; i += gridDim.x, ++n) {
    const int slot = n & 1;
    if (!mbar_wait_warp(&ifull[slot], (n >> 1) & 1, p.status)) return;
    const Item it = decode_item(i, p, info[2 * slot + 1]);
    const int head0 = it.h * p.G + it.hg * GC;
    const int flag = info[2 * slot];
    const bool bad = flag != 0;
    const uint32_t q_addr = smem_u32(q_ring + slot * GC * kQRow + dh * kQHalf);

    float m[GC], l[GC];
    float2 o[GC][4];
#pragma unroll
    for (int g = 0; g < GC; ++g) {
      m[g] = -INFINITY;
      l[g] = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) o[g][k] = make_float2(0.f, 0.f);
    }

    for (int pg = it.pg0; pg < it.pg1; ++pg) {
      const int nvalid = min(max(it.ctx - pg * kPage - kTokPerWarp * warp, 0), kTokPerWarp);
      // ---- K tile: scores, lane = (token t, dim half dh), 64 dims of row t
      if (!mbar_wait_warp(&full[rs], rph, p.status)) return;
      const uint32_t kb = smem_u32(smem + rs * kStageBytes);
      float2 acc[GC];
      if (nvalid > 0) {
        const int t = kTokPerWarp * warp + tq;
#pragma unroll
        for (int g = 0; g < GC; ++g) acc[g] = make_float2(0.f, 0.f);
        const uint32_t krow = kb + dh * kBoxBytes + t * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 kw = lds128(krow + ((c ^ (t & 7)) << 4));
          const float2 k0 = bf16x2_to_float2(kw.x), k1 = bf16x2_to_float2(kw.y);
          const float2 k2 = bf16x2_to_float2(kw.z), k3 = bf16x2_to_float2(kw.w);
#pragma unroll
          for (int g = 0; g < GC; ++g) {
            const float4 qa = lds128f(q_addr + (g * kQRow + c * 8) * 4);
            const float4 qb = lds128f(q_addr + (g * kQRow + c * 8 + 4) * 4);
            acc[g] = __ffma2_rn(make_float2(qa.x, qa.y), k0, acc[g]);
            acc[g] = __ffma2_rn(make_float2(qa.z, qa.w), k1, acc[g]);
            acc[g] = __ffma2_rn(make_float2(qb.x, qb.y), k2, acc[g]);
            acc[g] = __ffma2_rn(make_float2(qb.z, qb.w), k3, acc[g]);
          }
        }
      }
      if (nvalid > 0) {
        // ---- online softmax over the warp's 16 tokens (log2 domain)
        const bool tv = tq < nvalid;
#pragma unroll
        for (int g = 0; g < GC; ++g) {
          float sc = acc[g].x + acc[g].y;
          sc += __shfl_xor_sync(0xffffffffu, sc, 16);
          sc = tv ? sc : -INFINITY;
          float mx = sc;
#pragma unroll
          for (int off = 8; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
          const float mn = fmaxf(m[g], mx);  // finite: nvalid > 0
          const float pv = fast_exp2(sc - mn);
          if (mn != m[g]) {  // warp-uniform
            const float alpha = fast_exp2(m[g] - mn);
            l[g] *= alpha;
            const float2 aa = make_float2(alpha, alpha);
#pragma unroll
            for (int k = 0; k < 4; ++k) o[g][k] = __fmul2_rn(o[g][k], aa);
            m[g] = mn;
          }
          if (dh == 0) {
            l[g] += pv;
            *reinterpret_cast<float2*>(p_s + (warp * kTokPerWarp + tq) * L::PS + 2 * g) =
                make_float2(pv, pv);
          }
        }
        __syncwarp();
      }
      // ---- V tile: P.V, half-warp per token, lane owns dims 8*jd .. 8*jd+7
      if (nvalid > 0) {
        const uint32_t vrow = kb + 2 * kBoxBytes + (jd >> 3) * kBoxBytes;
        const int jc = jd & 7;
        auto pv_token = [&](int tl, bool active) {
          const int tt = kTokPerWarp * warp + tl;
          uint4 vw = lds128(vrow + tt * 128 + ((jc ^ (tt & 7)) << 4));
          if (!active) vw = make_uint4(0u, 0u, 0u, 0u);
          const float2 v0 = bf16x2_to_float2(vw.x), v1 = bf16x2_to_float2(vw.y);
          const float2 v2 = bf16x2_to_float2(vw.z), v3 = bf16x2_to_float2(vw.w);
          float2 pr[L::PS / 2];
#pragma unroll
          for (int g2 = 0; g2 < L::PS / 2; g2 += 2) {
            const float4 pq = lds128f(p_addr + (tl * L::PS + 2 * g2) * 4);
            pr[g2] = make_float2(pq.x, pq.y);
            pr[g2 + 1] = make_float2(pq.z, pq.w);
          }
#pragma unroll
          for (int g = 0; g < GC; ++g) {
            const float2 pp = pr[g];
            o[g][0] = __ffma2_rn(pp, v0, o[g][0]);
            o[g][1] = __ffma2_rn(pp, v1, o[g][1]);
            o[g][2] = __ffma2_rn(pp, v2, o[g][2]);
            o[g][3] = __ffma2_rn(pp, v3, o[g][3]);
          }
        };
        if (nvalid == kTokPerWarp) {
#pragma unroll
          for (int tt = 0; tt < kTokPerWarp; tt += 2) pv_token(tt + half, true);
        } else {
          for (int tt = 0; tt < nvalid; tt += 2) {
            const int tl = tt + half;
            pv_token(min(tl, kTokPerWarp - 1), tl < nvalid);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[rs]);  // page consumed
      if (++rs == kStages) { rs = 0; rph ^= 1; }
    }
    if (lane == 0) mbar_arrive(&iempty[slot]);  // done with the item slot

    // ---- publish this warp's state; one warp (rotating) merges while the
    //      others move on to the next item
#pragma unroll
    for (int g = 0; g < GC; ++g) {
#pragma unroll
      for (int off = 16; off; off >>= 1) l[g] += __shfl_xor_sync(0xffffffffu, l[g], off);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        o[g][k].x += __shfl_xor_sync(0xffffffffu, o[g][k].x, 16);
        o[g][k].y += __shfl_xor_sync(0xffffffffu, o[g][k].y, 16);
      }
    }
    if (!mbar_wait_warp(merge_free, (n & 1) ^ 1, p.status)) return;  // previous merge read
    if (half == 0) {
#pragma unroll
      for (int g = 0; g < GC; ++g) {
        float4* dst = reinterpret_cast<float4*>(m_o + (warp * GC + g) * kHeadDim + jd * 8);
        dst[0] = make_float4(o[g][0].x, o[g][0].y, o[g][1].x, o[g][1].y);
        dst[1] = make_float4(o[g][2].x, o[g][2].y, o[g][3].x, o[g][3].y);
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int g = 0; g < GC; ++g) {
        m_ml[(warp * GC + g) * 2] = m[g];
        m_ml[(warp * GC + g) * 2 + 1] = l[g];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(merge_ready);
    if (warp == (int)(n % kConsumerWarps)) {
      if (!mbar_wait_warp(merge_ready, n & 1, p.status)) return;
      if (bad && lane == 0 && p.status)
        atomicOr(p.status, flag == 1 ? PA_STATUS_BAD_PAGE : PA_STATUS_BAD_LENGTH);
      // lane owns dims 4*lane .. 4*lane+3 of every head of the group
      float4 res[GC];
      float lse[GC];
#pragma unroll
      for (int g = 0; g < GC; ++g) {
        float mw[kConsumerWarps], M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          mw[w] = m_ml[(w * GC + g) * 2];
          M = fmaxf(M, mw[w]);
        }
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float Lsum = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float sw = fast_exp2(mw[w] - M);
            Lsum = fmaf(m_ml[(w * GC + g) * 2 + 1], sw, Lsum);
            const float4 ow =
                *reinterpret_cast<const float4*>(m_o + (w * GC + g) * kHeadDim + 4 * lane);
            acc.x = fmaf(ow.x, sw, acc.x);
            acc.y = fmaf(ow.y, sw, acc.y);
            acc.z = fmaf(ow.z, sw, acc.z);
            acc.w = fmaf(ow.w, sw, acc.w);
          }
        }
        const bool zero = bad || Lsum == 0.f;
        const float inv = zero ? 0.f : 1.f / Lsum;
        res[g] = zero ? make_float4(0.f, 0.f, 0.f, 0.f)
                      : make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        lse[g] = bad ? INFINITY : (Lsum > 0.f ? (M + __log2f(Lsum)) * kLn2 : -INFINITY);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(merge_free);  // shared state consumed into registers
      const int64_t row0 = (int64_t)it.s * p.Hq + head0;
#pragma unroll
      for (int g = 0; g < GC; ++g) {
        const int64_t row = row0 + g;
        if (p.S == 1) {
          if (p.out_f32) {
            reinterpret_cast<float4*>(p.out)[row * (kHeadDim / 4) + lane] = res[g];
          } else {
            uint2 u;
            u.x = pack_bf16x2(res[g].x, res[g].y);
            u.y = pack_bf16x2(res[g].z, res[g].w);
            reinterpret_cast<uint2*>(p.out)[row * (kHeadDim / 4) + lane] = u;
          }
        } else {
          reinterpret_cast<float4*>(p.part_o)[(row * p.S + it.j) * (kHeadDim / 4) + lane] = res[g];
          if (lane == 0) p.part_lse[row * p.S + it.j] = lse[g];
        }
      }
    }
  }
}

template <int GC>
cudaError_t launch_gc(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const DecodeParams& p,
                      int num_sms, cudaStream_t stream) {
  using L = Layout<GC>;
  static_assert(L::alloc <= kSmemLimit, "decode shared memory exceeds the per-CTA limit");
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<GC>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::alloc);
  if (e != cudaSuccess) return e;
  int grid = p.num_items < num_sms ? p.num_items : num_sms;
  if (grid < 1) return cudaSuccess;
  decode_kernel<GC><<<grid, kThreads, L::alloc, stream>>>(tm_k, tm_v, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                          const DecodeParams& p, int gc, int num_sms, cudaStream_t stream) {
  switch (gc) {
    case 1: return launch_gc<1>(tm_k, tm_v, p, num_sms, stream);
    case 2: return launch_gc<2>(tm_k, tm_v, p, num_sms, stream);
    case 3: return launch_gc<3>(tm_k, tm_v, p, num_sms, stream);
    case 4: return launch_gc<4>(tm_k, tm_v, p, num_sms, stream);
    case 5: return launch_gc<5>(tm_k, tm_v, p, num_sms, stream);
    case 6: return launch_gc<6>(tm_k, tm_v, p, num_sms, stream);
    case 7: return launch_gc<7>(tm_k, tm_v, p, num_sms, stream);
    case 8: return launch_gc<8>(tm_k, tm_v, p, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
