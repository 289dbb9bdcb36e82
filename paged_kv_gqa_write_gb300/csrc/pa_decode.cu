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
//  * One producer warp streams each page's K and V tiles (128 tokens x 128
//    dims, 32 KB each) with 2-D TMA loads (two 64-column boxes per tile,
//    128-byte swizzle) into a 3-stage shared-memory ring guarded by mbarriers,
//    with an L2 evict-first policy (the cache is streamed once).
//  * Four consumer warps share each page: warp w owns tokens 32w..32w+31.
//    Scores: lane = token; the K row is read once from shared memory (swizzle
//    makes the 32 rows conflict-free) and used for all GC query heads, whose
//    pre-scaled FP32 values are broadcast from shared memory; products are
//    accumulated with packed FP32 FMAs (fma.rn.f32x2).
//    Softmax: per-warp running max by warp shuffles, exp2 with log2(e) folded
//    into the scale, per-lane partial sums.  P.V: a half-warp per token, each
//    lane owning 8 output dims; tokens past the context are skipped (a select
//    keeps poisoned tail rows out: 0 * NaN would be NaN).
//  * Item end: the four warps' (m, l, o) merge in shared memory in a fixed
//    order; the result goes to `out` (one split) or to normalised partials
//    (o, lse) that the combine kernel merges.
#include "pa_launch.cuh"

namespace pa {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 3;
constexpr int kBoxBytes = 64 * 2 * kPage;     // 64 dims x 128 tokens of bf16 = 16 KB
constexpr int kStageBytes = 4 * kBoxBytes;    // K lo, K hi, V lo, V hi
constexpr float kLn2 = 0.69314718055994530942f;

template <int GC>
struct Layout {
  static constexpr int PS = (GC + 3) & ~3;                      // p row stride (floats)
  static constexpr int q = kStages * kStageBytes;               // q_s [GC][128] f32
  static constexpr int p = q + GC * kHeadDim * 4;               // p_s [4][32][PS] f32
  static constexpr int mo = p + kConsumerWarps * 32 * PS * 4;   // merge o [4][GC][128]
  static constexpr int mml = mo + kConsumerWarps * GC * kHeadDim * 4;  // merge m,l [4][GC][2]
  static constexpr int bars = (mml + kConsumerWarps * GC * 2 * 4 + 7) & ~7;
  static constexpr int total = bars + 2 * kStages * 8;
  static constexpr int alloc = total + 1024;                    // room to align to 1024 B
};

struct Item {
  int s, h, hg, j, pg0, pg1, ctx;
  bool ok;
};

__device__ __forceinline__ Item decode_item(int i, const DecodeParams& p) {
  Item it;
  const int per_seq = p.Hkv * p.NG;
  const int U = p.B * per_seq;
  it.j = i / U;
  const int u = i - it.j * U;
  it.s = u / per_seq;
  const int r = u - it.s * per_seq;
  it.h = r / p.NG;
  it.hg = r - it.h * p.NG;
  it.ctx = __ldg(p.context_lens + it.s);
  it.ok = it.ctx >= 0 && it.ctx <= p.max_pages * kPage;
  const int npg = it.ok ? (it.ctx + kPage - 1) / kPage : 0;
  it.pg0 = it.j * p.pps;
  it.pg1 = min(npg, it.pg0 + p.pps);
  if (it.pg1 < it.pg0) it.pg1 = it.pg0;
  return it;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int GC>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  using L = Layout<GC>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::bars);
  uint64_t* empty = full + kStages;
  float* q_s = reinterpret_cast<float*>(smem + L::q);
  float* p_s = reinterpret_cast<float*>(smem + L::p);
  float* m_o = reinterpret_cast<float*>(smem + L::mo);
  float* m_ml = reinterpret_cast<float*>(smem + L::mml);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensor_map(&tm_k);
      prefetch_tensor_map(&tm_v);
      const uint64_t pol = l2_policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      for (int i = blockIdx.x; i < p.num_items; i += gridDim.x) {
        const Item it = decode_item(i, p);
        const int32_t* bt = p.block_table + (int64_t)it.s * p.max_pages;
        for (int pg = it.pg0; pg < it.pg1; ++pg) {
          int page = __ldg(bt + pg);
          if (page < 0 || page >= p.num_pages) page = 0;  // consumers flag and zero it
          if (!mbar_wait(&empty[stage], phase ^ 1, p.status)) return;
          mbar_arrive_expect_tx(&full[stage], kStageBytes);
          uint8_t* st = smem + stage * kStageBytes;
          const int x = it.h * kHeadDim, y = page * kPage;
          tma_load_2d(st, &tm_k, x, y, &full[stage], pol);
          tma_load_2d(st + kBoxBytes, &tm_k, x + 64, y, &full[stage], pol);
          tma_load_2d(st + 2 * kBoxBytes, &tm_v, x, y, &full[stage], pol);
          tma_load_2d(st + 3 * kBoxBytes, &tm_v, x + 64, y, &full[stage], pol);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int tid = threadIdx.x;  // 0..127
  const int half = lane >> 4, jd = lane & 15;  // P.V: token parity, 8-dim chunk
  const uint32_t q_addr = smem_u32(q_s);
  const uint32_t p_addr = smem_u32(p_s) + warp * 32 * L::PS * 4;
  int stage = 0;
  uint32_t phase = 0;
  bool aborted = false;

  for (int i = blockIdx.x; i < p.num_items && !aborted; i += gridDim.x) {
    const Item it = decode_item(i, p);
    const int head0 = it.h * p.G + it.hg * GC;
    {
      const __nv_bfloat16* qg = p.q + ((int64_t)it.s * p.Hq + head0) * kHeadDim;
#pragma unroll
      for (int g = 0; g < GC; ++g)
        q_s[g * kHeadDim + tid] = __bfloat162float(qg[g * kHeadDim + tid]) * p.scale_log2;
    }
    named_bar_sync(1, kConsumerWarps * 32);

    float m[GC], l[GC];
    float2 o[GC][4];
#pragma unroll
    for (int g = 0; g < GC; ++g) {
      m[g] = -INFINITY;
      l[g] = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) o[g][k] = make_float2(0.f, 0.f);
    }
    bool bad = !it.ok;
    const int32_t* bt = p.block_table + (int64_t)it.s * p.max_pages;

    for (int pg = it.pg0; pg < it.pg1; ++pg) {
      const int page = __ldg(bt + pg);
      bad |= (page < 0 || page >= p.num_pages);
      if (!mbar_wait_warp(&full[stage], phase, p.status)) { aborted = true; break; }
      const uint32_t kb = smem_u32(smem + stage * kStageBytes);
      const uint32_t vb = kb + 2 * kBoxBytes;
      const int nvalid = min(max(it.ctx - pg * kPage - 32 * warp, 0), 32);
      if (nvalid > 0) {
        // ---- scores: lane = token t of this warp's slice
        const int t = 32 * warp + lane;
        float2 acc[GC];
#pragma unroll
        for (int g = 0; g < GC; ++g) acc[g] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const uint32_t a = kb + (c >> 3) * kBoxBytes + t * 128 + (((c & 7) ^ (t & 7)) << 4);
          const uint4 kw = lds128(a);
          const float2 k0 = bf16x2_to_float2(kw.x), k1 = bf16x2_to_float2(kw.y);
          const float2 k2 = bf16x2_to_float2(kw.z), k3 = bf16x2_to_float2(kw.w);
#pragma unroll
          for (int g = 0; g < GC; ++g) {
            const float4 qa = lds128f(q_addr + (g * kHeadDim + c * 8) * 4);
            const float4 qb = lds128f(q_addr + (g * kHeadDim + c * 8 + 4) * 4);
            acc[g] = __ffma2_rn(make_float2(qa.x, qa.y), k0, acc[g]);
            acc[g] = __ffma2_rn(make_float2(qa.z, qa.w), k1, acc[g]);
            acc[g] = __ffma2_rn(make_float2(qb.x, qb.y), k2, acc[g]);
            acc[g] = __ffma2_rn(make_float2(qb.z, qb.w), k3, acc[g]);
          }
        }
        // ---- online softmax over this warp's tokens (log2 domain)
        const bool tv = lane < nvalid;
#pragma unroll
        for (int g = 0; g < GC; ++g) {
          const float sc = tv ? acc[g].x + acc[g].y : -INFINITY;
          const float mn = fmaxf(m[g], warp_max(sc));  // finite: nvalid > 0
          const float alpha = fast_exp2(m[g] - mn);
          const float pv = fast_exp2(sc - mn);
          l[g] = l[g] * alpha + pv;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            o[g][k].x *= alpha;
            o[g][k].y *= alpha;
          }
          m[g] = mn;
          p_s[warp * 32 * L::PS + lane * L::PS + g] = pv;
        }
        __syncwarp();
        // ---- P.V: half-warp per token, lane owns dims 8*jd .. 8*jd+7
        const uint32_t vrow = vb + (jd >> 3) * kBoxBytes;
        const int jc = jd & 7;
        auto pv_token = [&](int tl, bool active) {
          const int tt = 32 * warp + tl;
          uint4 vw = lds128(vrow + tt * 128 + ((jc ^ (tt & 7)) << 4));
          if (!active) vw = make_uint4(0u, 0u, 0u, 0u);
          const float2 v0 = bf16x2_to_float2(vw.x), v1 = bf16x2_to_float2(vw.y);
          const float2 v2 = bf16x2_to_float2(vw.z), v3 = bf16x2_to_float2(vw.w);
          float pr[L::PS];
#pragma unroll
          for (int g4 = 0; g4 < L::PS; g4 += 4) {
            const float4 pq = lds128f(p_addr + (tl * L::PS + g4) * 4);
            pr[g4] = pq.x;
            if (g4 + 1 < L::PS) pr[g4 + 1] = pq.y;
            if (g4 + 2 < L::PS) pr[g4 + 2] = pq.z;
            if (g4 + 3 < L::PS) pr[g4 + 3] = pq.w;
          }
#pragma unroll
          for (int g = 0; g < GC; ++g) {
            const float2 pp = make_float2(pr[g], pr[g]);
            o[g][0] = __ffma2_rn(pp, v0, o[g][0]);
            o[g][1] = __ffma2_rn(pp, v1, o[g][1]);
            o[g][2] = __ffma2_rn(pp, v2, o[g][2]);
            o[g][3] = __ffma2_rn(pp, v3, o[g][3]);
          }
        };
        if (nvalid == 32) {
#pragma unroll 4
          for (int tt = 0; tt < 32; tt += 2) pv_token(tt + half, true);
        } else {
          for (int tt = 0; tt < nvalid; tt += 2) {
            const int tl = tt + half;
            pv_token(min(tl, 31), tl < nvalid);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == kStages) { stage = 0; phase ^= 1; }
    }
    if (aborted) break;

    // ---- merge the four warps' states (fixed order) and write the result
#pragma unroll
    for (int g = 0; g < GC; ++g) {
      l[g] = warp_sum(l[g]);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        o[g][k].x += __shfl_xor_sync(0xffffffffu, o[g][k].x, 16);
        o[g][k].y += __shfl_xor_sync(0xffffffffu, o[g][k].y, 16);
      }
      if (half == 0) {
        float4* dst = reinterpret_cast<float4*>(m_o + (warp * GC + g) * kHeadDim + jd * 8);
        dst[0] = make_float4(o[g][0].x, o[g][0].y, o[g][1].x, o[g][1].y);
        dst[1] = make_float4(o[g][2].x, o[g][2].y, o[g][3].x, o[g][3].y);
      }
      if (lane == 0) {
        m_ml[(warp * GC + g) * 2] = m[g];
        m_ml[(warp * GC + g) * 2 + 1] = l[g];
      }
    }
    named_bar_sync(1, kConsumerWarps * 32);
    if (bad && tid == 0 && p.status)
      atomicOr(p.status, it.ok ? PA_STATUS_BAD_PAGE : PA_STATUS_BAD_LENGTH);
    const int d = tid;
#pragma unroll
    for (int g = 0; g < GC; ++g) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, m_ml[(w * GC + g) * 2]);
      float Lsum = 0.f, O = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float sw = fast_exp2(m_ml[(w * GC + g) * 2] - M);
          Lsum += m_ml[(w * GC + g) * 2 + 1] * sw;
          O += m_o[(w * GC + g) * kHeadDim + d] * sw;
        }
      }
      const float res = (bad || Lsum == 0.f) ? 0.f : O / Lsum;
      const int64_t row = (int64_t)it.s * p.Hq + head0 + g;
      if (p.S == 1) {
        if (p.out_f32)
          reinterpret_cast<float*>(p.out)[row * kHeadDim + d] = res;
        else
          reinterpret_cast<__nv_bfloat16*>(p.out)[row * kHeadDim + d] = __float2bfloat16_rn(res);
      } else {
        p.part_o[(row * p.S + it.j) * kHeadDim + d] = res;
        if (d == 0)
          p.part_lse[row * p.S + it.j] =
              bad ? INFINITY : (Lsum > 0.f ? (M + __log2f(Lsum)) * kLn2 : -INFINITY);
      }
    }
  }
}

template <int GC>
cudaError_t launch_gc(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const DecodeParams& p,
                      int num_sms, cudaStream_t stream) {
  using L = Layout<GC>;
  static_assert(L::alloc <= 232448, "decode shared memory exceeds the per-CTA limit");
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
