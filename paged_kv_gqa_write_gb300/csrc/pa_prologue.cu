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
// Memory bound and small (decode: B tokens): a warp takes a token and 8 of
// its Hq + 2 Hkv heads, resolves the token's slot and validity (as the KV
// write does) while those heads' rows load, computes the (cos, sin) pairs of
// its position -- the angle pos * base^(-2i/D) / scale reduced modulo 2 pi in
// double precision so that long contexts keep full accuracy -- and runs the
// heads.
// A lane holds 4 of a head's 128 values: the RMS is one warp reduction, and
// NeoX pairs (i, i+64) sit in lanes l and l+16, one shuffle apart.
#include "pa_launch.cuh"

namespace pa {
namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 8;  // heads per warp, all loaded before the token's slot is resolved

__device__ __forceinline__ float4 bf16x4_to_float4(uint2 w) {
  const float2 a = bf16x2_to_float2(w.x), b = bf16x2_to_float2(w.y);
  return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ uint2 float4_to_bf16x4(float4 v) {
  return make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
}

__global__ void __launch_bounds__(kThreads) prologue_kernel(const PrologueParams p) {
  extern __shared__ int32_t pro_smem[];
  int32_t* off = pro_smem;                                 // [B] chunk offsets
  int32_t* scratch = pro_smem + (p.chunk_lens ? p.B : 0);  // [kThreads]
  __shared__ double freq[64];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the 64 frequencies base^(-2i/D) / scale, once per CTA
  if (threadIdx.x < 64)
    freq[threadIdx.x] = exp2(-2.0 * threadIdx.x / kHeadDim * p.log2_base) / p.rope_scale;
  if (p.chunk_lens) {
    const bool neg = block_chunk_offsets(p.chunk_lens, p.B, off, scratch);
    if (blockIdx.x == 0 && threadIdx.x == 0 && p.status) {
      if (neg) atomicOr(p.status, PA_STATUS_BAD_LENGTH);
      if ((p.B > 0 ? off[p.B - 1] : 0) != p.T) atomicOr(p.status, PA_STATUS_BAD_TOKENS);
    }
  } else {
    __syncthreads();
  }
  const int heads = p.Hq + 2 * p.Hkv;
  const int chunks = (heads + kChunk - 1) / kChunk;  // head chunks per token
  const int64_t units = (int64_t)p.T * chunks;
  const int warps = gridDim.x * (kThreads / 32);
  // a warp per (token, chunk of kChunk heads); lane l holds values 4l .. 4l+3 of each head
  for (int64_t u = (int64_t)blockIdx.x * (kThreads / 32) + warp; u < units; u += warps) {
    const int token = (int)(u / chunks);
    const int h0 = (int)(u - (int64_t)token * chunks) * kChunk;
    const int h1 = min(heads, h0 + kChunk);
    const uint2* row = p.qkv + (int64_t)token * heads * (kHeadDim / 4);
    // the chunk's rows load while the token's slot is resolved
    uint2 raw[kChunk];
#pragma unroll
    for (int k = 0; k < kChunk; ++k)
      raw[k] = h0 + k < h1 ? __ldg(row + (h0 + k) * (kHeadDim / 4) + lane) : make_uint2(0u, 0u);
    int s, j, n;
    if (p.chunk_lens) {
      s = seq_of_token(off, p.B, token);
      j = s < p.B ? token - (s ? off[s - 1] : 0) : 0;
      n = s < p.B ? p.chunk_lens[s] : 0;
    } else {
      s = token;
      j = 0;
      n = 1;
    }
    int err = PA_STATUS_BAD_TOKENS;  // a token past sum(chunk_lens): flagged above
    int ctx = 0;
    if (s < p.B) {
      ctx = p.context_lens[s];
      err = warp_check_sequence(p.block_table, s, ctx, n, p.num_pages, p.max_pages);
      if (err && lane == 0 && p.status) atomicOr(p.status, err);
    }
    const bool valid = err == 0;
    const int pos = valid ? ctx - n + j : 0;
    const int64_t slot =
        valid ? (int64_t)p.block_table[(int64_t)s * p.max_pages + pos / kPage] * kPage + pos % kPage
              : 0;
    // angles of pairs lane and lane + 32: pos * f_i reduced to [-pi, pi] in
    // double precision (three operations; long contexts reach thousands of
    // radians), then the single-precision sine and cosine of the remainder
    constexpr double kTwoPi = 6.283185307179586476925286766559;
    float c_lo, s_lo, c_hi, s_hi;
    {
      const double a0 = (double)pos * freq[lane], a1 = (double)pos * freq[lane + 32];
      sincosf((float)fma(-rint(a0 * (1.0 / kTwoPi)), kTwoPi, a0), &s_lo, &c_lo);
      sincosf((float)fma(-rint(a1 * (1.0 / kTwoPi)), kTwoPi, a1), &s_hi, &c_hi);
    }
    // this lane's values 4l .. 4l+3 belong to pair (4l .. 4l+3) mod 64
    const int i0 = (lane & 15) * 4;
    float cq[4], sq[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = i0 + e;
      const float cl = __shfl_sync(0xffffffffu, c_lo, i & 31);
      const float ch = __shfl_sync(0xffffffffu, c_hi, i & 31);
      const float sl = __shfl_sync(0xffffffffu, s_lo, i & 31);
      const float sh = __shfl_sync(0xffffffffu, s_hi, i & 31);
      cq[e] = i < 32 ? cl : ch;
      sq[e] = (i < 32 ? sl : sh) * (lane < 16 ? -1.f : 1.f);
    }
#pragma unroll
    for (int k = 0; k < kChunk; ++k) {
      const int hh = h0 + k;
      if (hh >= h1) break;
      const uint2 w4 = raw[k];
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
      const float4 w = __ldg(reinterpret_cast<const float4*>(is_q ? p.wq : p.wk) + lane);
      const float4 y = make_float4(x.x * r * w.x, x.y * r * w.y, x.z * r * w.z, x.w * r * w.w);
      // NeoX pairs (i, i + 64): lane l < 16 holds the first halves, l + 16 the second
      const float4 z = make_float4(__shfl_xor_sync(0xffffffffu, y.x, 16),
                                   __shfl_xor_sync(0xffffffffu, y.y, 16),
                                   __shfl_xor_sync(0xffffffffu, y.z, 16),
                                   __shfl_xor_sync(0xffffffffu, y.w, 16));
      const float4 o = make_float4(fmaf(sq[0], z.x, y.x * cq[0]), fmaf(sq[1], z.y, y.y * cq[1]),
                                   fmaf(sq[2], z.z, y.z * cq[2]), fmaf(sq[3], z.w, y.w * cq[3]));
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
  }
}

}  // namespace

cudaError_t launch_prologue(const PrologueParams& p, int num_sms, cudaStream_t stream) {
  if (p.T <= 0) return cudaSuccess;
  const int64_t units = (int64_t)p.T * ((p.Hq + 2 * p.Hkv + kChunk - 1) / kChunk);
  int64_t blocks64 = (units + kThreads / 32 - 1) / (kThreads / 32);
  int blocks = (int)(blocks64 < INT32_MAX ? blocks64 : INT32_MAX);
  const int cap = num_sms * 8;
  if (blocks > cap) blocks = cap;
  const size_t smem = p.chunk_lens ? (size_t)(p.B + kThreads) * sizeof(int32_t) : 0;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(prologue_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  prologue_kernel<<<blocks, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
