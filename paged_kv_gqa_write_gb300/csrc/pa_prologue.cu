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
// compute warps take the staged token's Q and K heads, two per warp at a time,
// and write the results with coalesced stores; the V rows leave the stage with
// one bulk store.  Rows in flight per SM (the ring depth times the resident
// CTAs) cover the HBM latency.
//
// The host computes the 64 frequencies in double precision.  The angle is
// carried in turns (angle / 2 pi): pos times the frequency in turns as an
// unevaluated float pair, whose product is exact up to the low
// word's rounding, so the whole turns drop out exactly and the remainder in
// [-1/2, 1/2] goes to sincospif.  Single precision throughout (the GPU's
// double-precision rate is a small fraction of its float rate); positions
// whose turn count leaves too few fraction bits take a double-precision path.
//
// A compute lane holds 8 of a head's 128 values, both members of four NeoX
// pairs (i, i+64): the RMS is a 16-lane reduction and the rotation needs no
// data from other lanes.
//
// Over an FP8 (e4m3) cache the same kernel quantizes what it stores: each K
// value as the BF16 cache would hold it (rounded to bf16), and each V value
// as given, divided by its KV head's scale (an FP32 quotient) and rounded to
// the nearest e4m3 code, saturating -- the bytes pa_kv_write_fp8 would write
// from those rows (an "fp8_e4m3" KV cache, "Qwen4-Exp QSA" blog, DGX Spark
// note).  V then leaves through the compute warps instead of a bulk store.
#include <cuda_fp8.h>

#include "pa_launch.cuh"

namespace pa {
namespace {

constexpr int kComputeWarps = 8;
constexpr int kThreads = (kComputeWarps + 1) * 32;  // warp 0: loader
constexpr int kMaxStages = 4;
constexpr int kStageBudget = 200 * 1024;            // shared memory for the row ring

// per stage: the token's cache slot (-1: invalid sequence, nothing written)
// and the cos / sin of its 64 rotary pairs
struct StageInfo {
  long long slot;
  int32_t valid, pad;
  float cs[2][64];
};

// 4 bf16 values over s -> 4 e4m3 codes (round to nearest even, saturating),
// value i in byte i.
__device__ __forceinline__ uint32_t quant4_e4m3(uint2 w, float s) {
  const float2 a = bf16x2_to_float2(w.x), b = bf16x2_to_float2(w.y);
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(a.x, s), __fdiv_rn(a.y, s)),
                                               __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(b.x, s), __fdiv_rn(b.y, s)),
                                               __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
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

template <bool FP8>
__global__ void __launch_bounds__(kThreads, 3)
    prologue_kernel(const __grid_constant__ PrologueParams p, int per_cta, int stages) {
  // an attention kernel launched next as a programmatic dependent may set up
  // meanwhile; it reads nothing before this grid has completed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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
      // angles of pairs lane and lane + 32, reduced to [-1/2, 1/2] turns (pos
      // exact in a float and pos * g < 2^22 turns: hi - rint(hi) is exact and
      // the fraction keeps at least 2^-24 resolution; very long positions: the
      // product and its reduction in double precision)
      float c_lo, s_lo, c_hi, s_hi;
      auto angles = [&](bool fast) {
        rope_sincos(pos, fast, turn_hi[lane], turn_lo[lane], freq[lane], s_lo, c_lo);
        rope_sincos(pos, fast, turn_hi[lane + 32], turn_lo[lane + 32], freq[lane + 32], s_hi, c_hi);
      };
      if (rope_fast(pos, gmax)) angles(true); else angles(false);
      in.cs[0][lane] = c_lo;
      in.cs[0][lane + 32] = c_hi;
      in.cs[1][lane] = s_lo;
      in.cs[1][lane + 32] = s_hi;
      mbar_arrive(&full[st]);  // with the row's bytes, completes the stage
    }
  } else {
    // ------------------------------------------------------------ compute
    // Half-warp h of a warp takes head 2m + h of the token's Q and K heads
    // (pair m = cw, cw + 8, ...).  Its lane li holds values i0 .. i0+3 and
    // i0+64 .. i0+67 (i0 = 4 li): each NeoX pair (i, i + 64) in one lane.
    const int cw = warp - 1, hl = lane >> 4, li = lane & 15, i0 = 4 * li;
    const float4 wq_lo = __ldg(reinterpret_cast<const float4*>(p.wq + i0));
    const float4 wq_hi = __ldg(reinterpret_cast<const float4*>(p.wq + i0 + 64));
    const float4 wk_lo = __ldg(reinterpret_cast<const float4*>(p.wk + i0));
    const float4 wk_hi = __ldg(reinterpret_cast<const float4*>(p.wk + i0 + 64));
    const int nqk = p.Hq + p.Hkv;
    for (int token = t0, i = 0; token < t1; ++token, ++i) {
      const int st = i % stages;
      if (!mbar_wait_warp(&full[st], (i / stages) & 1, p.status)) break;
      const StageInfo& in = info[st];
      const long long slot = in.slot;
      const bool valid = in.valid != 0;
      const uint8_t* row = rows + st * row_bytes;
      // V is copied bit for bit: one bulk store of the token's Hkv V rows,
      // which are contiguous in the staged row and in the cache slot
      const bool v_store = !FP8 && cw == 0 && lane == 0 && valid;
      if (v_store) {
        asm volatile(
            "cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n\t"
            "cp.async.bulk.commit_group;" ::"l"(reinterpret_cast<uint64_t>(
                reinterpret_cast<uint8_t*>(p.v_cache) + slot * p.Hkv * (kHeadDim * 2))),
            "r"(smem_u32(row + nqk * (kHeadDim * 2))), "r"((uint32_t)p.Hkv * (kHeadDim * 2))
            : "memory");
      }
      const float4 c4 = *reinterpret_cast<const float4*>(&in.cs[0][i0]);
      const float4 s4 = *reinterpret_cast<const float4*>(&in.cs[1][i0]);
      for (int m = cw; 2 * m < nqk; m += kComputeWarps) {
        const int hh = 2 * m + hl;
        const bool live = hh < nqk;
        const uint8_t* hrow = row + (live ? hh : 0) * (kHeadDim * 2);
        const uint2 ra = *reinterpret_cast<const uint2*>(hrow + 8 * li);
        const uint2 rb = *reinterpret_cast<const uint2*>(hrow + 128 + 8 * li);
        const bool is_q = hh < p.Hq;
        float4 oa, ob;
        norm_rope_half(ra, rb, is_q ? wq_lo : wk_lo, is_q ? wq_hi : wk_hi, c4, s4, p.eps,
                       is_q ? p.q_scale : 1.f, oa, ob);
        if (!live) continue;
        uint2* dst;
        if (is_q) {
          dst = p.q_out + ((int64_t)token * p.Hq + hh) * (kHeadDim / 4);
        } else {
          if (!valid) continue;
          if constexpr (FP8) {
            // K as the bf16 cache would hold it, over the head's scale
            const int h = hh - p.Hq;
            const float ks = __ldg(p.k_scale + h);
            uint32_t* kd = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(p.k_cache) +
                                                       (slot * p.Hkv + h) * kHeadDim);
            kd[li] = quant4_e4m3(float4_to_bf16x4(oa), ks);
            kd[16 + li] = quant4_e4m3(float4_to_bf16x4(ob), ks);
            continue;
          }
          dst = p.k_cache + (slot * p.Hkv + (hh - p.Hq)) * (kHeadDim / 4);
        }
        // (an invalid sequence's Q rows are zero, like its attention output)
        dst[li] = valid ? float4_to_bf16x4(oa) : make_uint2(0u, 0u);
        dst[16 + li] = valid ? float4_to_bf16x4(ob) : make_uint2(0u, 0u);
      }
      if constexpr (FP8) {
        // V heads over their scales: half-warp per head, lane li values 8 li .. 8 li + 7
        if (valid) {
          for (int m = cw; 2 * m < p.Hkv; m += kComputeWarps) {
            const int h = 2 * m + hl;
            if (h >= p.Hkv) continue;
            const uint4 r = *reinterpret_cast<const uint4*>(row + (nqk + h) * (kHeadDim * 2) + 16 * li);
            const float vs = __ldg(p.v_scale + h);
            *reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(p.v_cache) +
                                      (slot * p.Hkv + h) * kHeadDim + 8 * li) =
                make_uint2(quant4_e4m3(make_uint2(r.x, r.y), vs), quant4_e4m3(make_uint2(r.z, r.w), vs));
          }
        }
      }
      // the V store must have read the stage before it is refilled
      if (v_store) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    // the V stores complete before the CTA exits
    if (cw == 0 && lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
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
  const bool fp8 = p.k_scale != nullptr;
  e = fp8 ? cudaFuncSetAttribute(prologue_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem)
          : cudaFuncSetAttribute(prologue_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
  if (e != cudaSuccess) return e;
  // resident CTAs per SM by shared memory (at most the 3 the registers allow)
  int per_sm = (int)((228 * 1024) / (smem + 2048));
  if (per_sm > 3) per_sm = 3;
  if (per_sm < 1) per_sm = 1;
  const int64_t slots = (int64_t)num_sms * per_sm;
  const int per_cta = (int)((p.T + slots - 1) / slots);
  const int blocks = (p.T + per_cta - 1) / per_cta;
  if (fp8)
    prologue_kernel<true><<<blocks, kThreads, smem, stream>>>(p, per_cta, stages);
  else
    prologue_kernel<false><<<blocks, kThreads, smem, stream>>>(p, per_cta, stages);
  return cudaGetLastError();
}

}  // namespace pa
