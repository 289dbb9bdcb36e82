// pa_prologue.cu -- the decode / prefill prologue: per-head RMSNorm of Q and
// K, NeoX rotary embedding at each new token's position, and the KV cache
// write, in one pass over the fused QKV projection output.
//
// "Qwen 3" (TensorSharp), section 3 "Forward graph": per-head RMSNorm(Q) and
// RMSNorm(K) with attn_q_norm / attn_k_norm weights, RoPE_NeoX(Q, K) at the
// tokens' positions, Q times 1/sqrt(headDim), then (K, V) appended to the
// cache; section 4.1: QK-norm over each head's headDim values, NeoX RoPE with
// frequencies from rope.freq_base and rope.scale (section 5: a frequency scale
// divisor); section 4.3: epsilon from the config.  "Qwen3-14B" (pypto-lib),
// "Model structure, top down": decode_fwd runs Q/K norm -> RoPE before the KV
// cache write; FP32 RMSNorm weights.
//
// Memory bound: each token's fused QKV row (Hq + 2 Hkv heads of 256 bytes,
// contiguous) is read once and Q, K and V rows are written once.  A CTA takes
// a contiguous run of tokens.  Its loader warp streams each token's row into a
// ring of shared-memory stages with one bulk copy, and while the copy is in
// flight it resolves the token's sequence, validity and cache slot and the
// (cos, sin) pairs of its position -- once per token, for all heads.  Eight
// compute warps take the heads of the staged token (head w, w + 8, ...) and
// write the results with coalesced stores.  Rows in flight per SM (the ring
// depth times the resident CTAs) cover the HBM latency.
//
// The host computes the 64 frequencies in double precision.  The angle is
// carried in turns (angle / 2 pi): pos times the frequency in turns as an
// unevaluated float pair, whose product is exact up to the low
// word's rounding, so the whole turns drop out exactly and the remainder in
// [-1/2, 1/2] goes to sincospif.  Single precision throughout (the GPU's
// double-precision rate is a small fraction of its float rate); positions
// whose turn count leaves too few fraction bits take a double-precision path.
//
// A compute lane holds 4 of a head's 128 values: the RMS is one warp
// reduction, and NeoX pairs (i, i+64) sit in lanes l and l+16, one shuffle
// apart.
#include "pa_launch.cuh"

namespace pa {
namespace {

constexpr int kComputeWarps = 8;
constexpr int kThreads = (kComputeWarps + 1) * 32;  // warp 0: loader
constexpr int kMaxStages = 4;
constexpr int kStageBudget = 200 * 1024;            // shared memory for the row ring
constexpr double kTwoPi = 6.283185307179586476925286766559;

// per stage: the token's cache slot (-1: invalid sequence, nothing written)
// and the cos / sin of its 64 rotary pairs
struct StageInfo {
  long long slot;
  int32_t valid, pad;
  float cs[2][64];
};

__device__ __forceinline__ float4 bf16x4_to_float4(uint2 w) {
  const float2 a = bf16x2_to_float2(w.x), b = bf16x2_to_float2(w.y);
  return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ uint2 float4_to_bf16x4(float4 v) {
  return make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// contiguous global -> shared bulk copy (16-byte aligned, a multiple of 16 bytes)
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__global__ void __launch_bounds__(kThreads, 3)
    prologue_kernel(const __grid_constant__ PrologueParams p, int per_cta, int stages) {
  extern __shared__ __align__(16) uint8_t pro_smem[];
  const int heads = p.Hq + 2 * p.Hkv;
  const uint32_t row_bytes = (uint32_t)heads * (kHeadDim * 2);
  uint8_t* rows = pro_smem;                                           // [stages][row_bytes]
  StageInfo* info = reinterpret_cast<StageInfo*>(rows + stages * row_bytes);  // [stages]
  uint64_t* full = reinterpret_cast<uint64_t*>(info + stages);        // [stages]
  uint64_t* empty = full + stages;                                    // [stages]
  int32_t* off = reinterpret_cast<int32_t*>(empty + stages);          // [B] chunk offsets
  int32_t* scratch = off + (p.chunk_lens ? p.B : 0);                  // [kThreads]
  __shared__ double freq[64];                 // base^(-2i/D) / scale, radians per position
  __shared__ float turn_hi[64], turn_lo[64];  // the same in turns, as hi + lo floats
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < 64) {
    freq[threadIdx.x] = p.freq[threadIdx.x];
    turn_hi[threadIdx.x] = p.turn_hi[threadIdx.x];
    turn_lo[threadIdx.x] = p.turn_lo[threadIdx.x];
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(&full[i], 32);
      mbar_init(&empty[i], kComputeWarps);
    }
    fence_mbar_init();
  }
  if (p.chunk_lens) {
    const bool neg = block_chunk_offsets(p.chunk_lens, p.B, off, scratch);
    if (blockIdx.x == 0 && threadIdx.x == 0 && p.status) {
      if (neg) atomicOr(p.status, PA_STATUS_BAD_LENGTH);
      if ((p.B > 0 ? off[p.B - 1] : 0) != p.T) atomicOr(p.status, PA_STATUS_BAD_TOKENS);
    }
  } else {
    __syncthreads();
  }
  const int t0 = blockIdx.x * per_cta, t1 = min(p.T, t0 + per_cta);

  if (warp == 0) {
    // ------------------------------------------------------------ loader
    const uint64_t pol = l2_policy_evict_first();  // each row is read once
    const float gmax = fmaxf(turn_hi[0], turn_hi[63]);  // the frequencies are monotone in i
    int last_s = -1, last_err = 0, last_ctx = 0, last_n = 0, pg = 0;
    for (int token = t0, i = 0; token < t1; ++token, ++i) {
      const int st = i % stages;
      if (!mbar_wait_warp(&empty[st], ((i / stages) & 1) ^ 1, p.status)) break;
      if (lane == 0) {
        mbar_expect_tx(&full[st], row_bytes);
        bulk_load(rows + st * row_bytes, reinterpret_cast<const uint8_t*>(p.qkv) +
                  (int64_t)token * row_bytes, row_bytes, &full[st], pol);
      }
      // the token's sequence and offset in its chunk
      int s, j;
      if (p.chunk_lens) {
        s = seq_of_token(off, p.B, token);
        j = s < p.B ? token - (s ? off[s - 1] : 0) : 0;
      } else {
        s = token;
        j = 0;
      }
      const int32_t* bt = p.block_table + (int64_t)s * p.max_pages;
      if (s < p.B && s != last_s) {
        // a new sequence: its length and first 32 block-table entries load
        // together; then lengths and every referenced entry are checked
        last_s = s;
        last_n = p.chunk_lens ? off[s] - (s ? off[s - 1] : 0) : 1;
        last_ctx = p.context_lens[s];
        pg = lane < p.max_pages ? bt[lane] : 0;
        const int ctx = last_ctx, n = last_n;
        if (ctx < 0 || n > ctx || ctx > p.max_pages * kPage) {
          last_err = PA_STATUS_BAD_LENGTH;
        } else {
          const int used = (ctx + kPage - 1) / kPage;
          bool bad = lane < used && (pg < 0 || pg >= p.num_pages);
          for (int e = lane + 32; e < used; e += 32) {
            const int q = bt[e];
            bad |= (q < 0 || q >= p.num_pages);
          }
          last_err = __any_sync(0xffffffffu, bad) ? PA_STATUS_BAD_PAGE : 0;
        }
        if (last_err && lane == 0 && p.status) atomicOr(p.status, last_err);
      }
      // a token past sum(chunk_lens) (flagged above) is invalid
      const bool valid = s < p.B && last_err == 0;
      const int pos = valid ? last_ctx - last_n + j : 0;
      // the slot's page: from the entries loaded with the sequence when among them
      const int pi = pos / kPage;
      const int page_sh = __shfl_sync(0xffffffffu, pg, pi & 31);
      StageInfo& in = info[st];
      if (lane == 0) {
        const int page = pi < 32 ? page_sh : (valid ? bt[pi] : 0);
        in.slot = valid ? (long long)page * kPage + pos % kPage : -1ll;
        in.valid = valid;
      }
      // angles of pairs lane and lane + 32, reduced to [-1/2, 1/2] turns
      float c_lo, s_lo, c_hi, s_hi;
      const float fpos = (float)pos;
      if (pos < (1 << 24) && fpos * gmax < 4194304.f) {
        // pos is exact in a float and pos * g < 2^22 turns: hi - rint(hi) is
        // exact and the fraction keeps at least 2^-24 resolution
        auto frac = [&](int q) {
          const float hi = fpos * turn_hi[q];
          const float lo = fmaf(fpos, turn_lo[q], fmaf(fpos, turn_hi[q], -hi));
          return (hi - rintf(hi)) + lo;
        };
        sincospif(2.f * frac(lane), &s_lo, &c_lo);
        sincospif(2.f * frac(lane + 32), &s_hi, &c_hi);
      } else {
        // very long positions: the product and its reduction in double precision
        const double a0 = (double)pos * freq[lane], a1 = (double)pos * freq[lane + 32];
        sincosf((float)fma(-rint(a0 * (1.0 / kTwoPi)), kTwoPi, a0), &s_lo, &c_lo);
        sincosf((float)fma(-rint(a1 * (1.0 / kTwoPi)), kTwoPi, a1), &s_hi, &c_hi);
      }
      in.cs[0][lane] = c_lo;
      in.cs[0][lane + 32] = c_hi;
      in.cs[1][lane] = s_lo;
      in.cs[1][lane + 32] = s_hi;
      mbar_arrive(&full[st]);  // with the row's bytes, completes the stage
    }
  } else {
    // ------------------------------------------------------------ compute
    const int cw = warp - 1;
    const float4 wq = __ldg(reinterpret_cast<const float4*>(p.wq) + lane);
    const float4 wk = __ldg(reinterpret_cast<const float4*>(p.wk) + lane);
    const int i0 = (lane & 15) * 4;  // this lane's values 4l .. 4l+3 belong to pairs i0 .. i0+3
    const float sgn = lane < 16 ? -1.f : 1.f;
    for (int token = t0, i = 0; token < t1; ++token, ++i) {
      const int st = i % stages;
      if (!mbar_wait_warp(&full[st], (i / stages) & 1, p.status)) break;
      const StageInfo& in = info[st];
      const long long slot = in.slot;
      const bool valid = in.valid != 0;
      const float4 cq = *reinterpret_cast<const float4*>(&in.cs[0][i0]);
      float4 sq = *reinterpret_cast<const float4*>(&in.cs[1][i0]);
      sq = make_float4(sq.x * sgn, sq.y * sgn, sq.z * sgn, sq.w * sgn);
      const uint2* row = reinterpret_cast<const uint2*>(rows + st * row_bytes);
      for (int hh = cw; hh < heads; hh += kComputeWarps) {
        const uint2 w4 = row[hh * (kHeadDim / 4) + lane];
        if (hh >= p.Hq + p.Hkv) {  // V: copied bit for bit
          if (valid) p.v_cache[(slot * p.Hkv + (hh - p.Hq - p.Hkv)) * (kHeadDim / 4) + lane] = w4;
          continue;
        }
        const bool is_q = hh < p.Hq;
        const float4 x = bf16x4_to_float4(w4);
        float ss = x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
#pragma unroll
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float r = rsqrtf(ss * (1.f / kHeadDim) + p.eps);
        const float4 w = is_q ? wq : wk;
        const float4 y = make_float4(x.x * r * w.x, x.y * r * w.y, x.z * r * w.z, x.w * r * w.w);
        // NeoX pairs (i, i + 64): lane l < 16 holds the first halves, l + 16 the second
        const float4 z = make_float4(__shfl_xor_sync(0xffffffffu, y.x, 16),
                                     __shfl_xor_sync(0xffffffffu, y.y, 16),
                                     __shfl_xor_sync(0xffffffffu, y.z, 16),
                                     __shfl_xor_sync(0xffffffffu, y.w, 16));
        const float4 o = make_float4(fmaf(sq.x, z.x, y.x * cq.x), fmaf(sq.y, z.y, y.y * cq.y),
                                     fmaf(sq.z, z.z, y.z * cq.z), fmaf(sq.w, z.w, y.w * cq.w));
        if (is_q) {
          // (an invalid sequence's rows are zero, like its attention output)
          const float qs = p.q_scale;
          p.q_out[((int64_t)token * p.Hq + hh) * (kHeadDim / 4) + lane] =
              valid ? float4_to_bf16x4(make_float4(o.x * qs, o.y * qs, o.z * qs, o.w * qs))
                    : make_uint2(0u, 0u);
        } else if (valid) {
          p.k_cache[(slot * p.Hkv + (hh - p.Hq)) * (kHeadDim / 4) + lane] = float4_to_bf16x4(o);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
  }
}

}  // namespace

cudaError_t launch_prologue(const PrologueParams& p, int num_sms, cudaStream_t stream) {
  if (p.T <= 0) return cudaSuccess;
  const size_t row_bytes = (size_t)(p.Hq + 2 * p.Hkv) * kHeadDim * 2;
  int stages = (int)(kStageBudget / (row_bytes + sizeof(StageInfo)));
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 1) stages = 1;
  const size_t smem = stages * (row_bytes + sizeof(StageInfo) + 2 * sizeof(uint64_t)) +
                      (p.chunk_lens ? (size_t)(p.B + kThreads) * sizeof(int32_t) : 0);
  int max_smem = 0, dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  if (smem + 2048 > (size_t)max_smem) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(prologue_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  // resident CTAs per SM by shared memory (at most the 3 the registers allow)
  int per_sm = (int)((228 * 1024) / (smem + 2048));
  if (per_sm > 3) per_sm = 3;
  if (per_sm < 1) per_sm = 1;
  const int64_t slots = (int64_t)num_sms * per_sm;
  const int per_cta = (int)((p.T + slots - 1) / slots);
  const int blocks = (p.T + per_cta - 1) / per_cta;
  prologue_kernel<<<blocks, kThreads, smem, stream>>>(p, per_cta, stages);
  return cudaGetLastError();
}

}  // namespace pa
