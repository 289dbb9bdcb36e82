// pa_kv_write.cu -- scatter the new tokens' K/V rows into the paged cache.
//
// "Qwen3-14B" (pypto-lib), "Model structure, top down": the KV cache write
// (decode) / KV cache update (prefill) precedes attention.  "Qwen 3"
// (TensorSharp), section 11: ScatterKv writes each token at slot
// blockId * blockSize + offset.  A pure byte copy, bound by launch latency at
// decode sizes and by HBM at prefill sizes: one warp per token moves the
// token's Hkv*256-byte K row and V row with 16-byte accesses, issuing the row
// loads before it resolves the token's slot so the two latencies overlap.
//
// The FP8 variant quantizes instead of copying (an "fp8_e4m3" KV cache, as in
// the SGLang measurement quoted by the "Qwen4-Exp QSA trafia na Ascend..."
// blog): element d of KV head h becomes the e4m3 code of x / scale[h] -- the
// FP32 quotient rounded to nearest, ties to even, saturating at +-448 -- so a
// token row shrinks to Hkv * 128 bytes.
#include <cuda_fp8.h>

#include "pa_launch.cuh"

namespace pa {

// 16 bf16 values (two 16-byte chunks) divided by s -> 16 e4m3 codes.
__device__ __forceinline__ uint4 quantize16(uint4 a, uint4 b, float s) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t r = 0;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint32_t x = w[2 * i + k];
      float2 f;
      f.x = __fdiv_rn(__uint_as_float(x << 16), s);
      f.y = __fdiv_rn(__uint_as_float(x & 0xffff0000u), s);
      const __nv_fp8x2_storage_t q = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
      r |= (uint32_t)q << (16 * k);
    }
    o[i] = r;
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

template <bool FP8>
__global__ void __launch_bounds__(256) kv_write_kernel(KvWriteParams p) {
  // an attention kernel launched next as a programmatic dependent may set up
  // meanwhile; it reads nothing before this grid has completed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ int32_t kvw_smem[];
  int32_t* off = kvw_smem;              // [B] when chunk_lens != null
  int32_t* scratch = kvw_smem + (p.chunk_lens ? p.B : 0);
  const int lane = threadIdx.x & 31;
  if (p.chunk_lens) {
    bool neg = block_chunk_offsets(p.chunk_lens, p.B, off, scratch);
    if (blockIdx.x == 0 && threadIdx.x == 0 && p.status) {
      if (neg) atomicOr(p.status, PA_STATUS_BAD_LENGTH);
      if ((p.B > 0 ? off[p.B - 1] : 0) != p.T) atomicOr(p.status, PA_STATUS_BAD_TOKENS);
    }
  }
  const int warps_per_block = blockDim.x >> 5;
  const int row_chunks = p.Hkv * (kHeadDim * 2 / 16);  // 16-byte chunks per token row
  // output chunks per row: a bf16 chunk is copied, an FP8 chunk takes two inputs
  const int out_chunks = FP8 ? row_chunks / 2 : row_chunks;
  constexpr int kIn = FP8 ? 2 : 1;   // input chunks per output chunk
  constexpr int kU = FP8 ? 2 : 4;    // output chunks per lane in flight
  for (int token = blockIdx.x * warps_per_block + (threadIdx.x >> 5); token < p.T;
       token += gridDim.x * warps_per_block) {
    const uint4* ks = p.k_new + (int64_t)token * row_chunks;
    const uint4* vs = p.v_new + (int64_t)token * row_chunks;
    int64_t slot = -1;  // resolved while the first rows load
    for (int c0 = 0; c0 < out_chunks; c0 += 32 * kU) {
      uint4 a[kU][kIn], b[kU][kIn];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < out_chunks) {
#pragma unroll
          for (int e = 0; e < kIn; ++e) {
            a[u][e] = __ldg(ks + kIn * c + e);
            b[u][e] = __ldg(vs + kIn * c + e);
          }
        }
      }
      if (c0 == 0) {
        int s, j, n;
        if (p.chunk_lens) {
          s = seq_of_token(off, p.B, token);
          if (s >= p.B) break;  // more tokens than sum(chunk_lens): flagged above
          j = token - (s ? off[s - 1] : 0);
          n = off[s] - (s ? off[s - 1] : 0);  // the token's sequence has n >= 1 tokens
        } else {
          s = token;
          j = 0;
          n = 1;
        }
        // the context length and the first 32 block-table entries load together
        const int32_t* bt = p.block_table + (int64_t)s * p.max_pages;
        const int ctx = p.context_lens[s];
        const int pg = lane < p.max_pages ? bt[lane] : 0;
        int err = 0;
        if (ctx < 0 || n > ctx || ctx > p.max_pages * kPage) {
          err = PA_STATUS_BAD_LENGTH;
        } else {
          const int used = (ctx + kPage - 1) / kPage;
          bool bad = lane < used && (pg < 0 || pg >= p.num_pages);
          for (int e = lane + 32; e < used; e += 32) {
            const int q = bt[e];
            bad |= (q < 0 || q >= p.num_pages);
          }
          err = __any_sync(0xffffffffu, bad) ? PA_STATUS_BAD_PAGE : 0;
        }
        if (err) {
          if (lane == 0 && p.status) atomicOr(p.status, err);
          break;
        }
        const int pos = ctx - n + j;
        const int pi = pos / kPage;
        const int page_sh = __shfl_sync(0xffffffffu, pg, pi & 31);
        const int page = pi < 32 ? page_sh : bt[pi];
        slot = (int64_t)page * kPage + pos % kPage;
      }
      uint4* kd = p.k_cache + slot * out_chunks;
      uint4* vd = p.v_cache + slot * out_chunks;
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < out_chunks) {
          if constexpr (FP8) {
            // 16 elements (32 input bytes, 16 output bytes) per chunk
            const int h = c / (kHeadDim / 16);
            kd[c] = quantize16(a[u][0], a[u][1], __ldg(p.k_scale + h));
            vd[c] = quantize16(b[u][0], b[u][1], __ldg(p.v_scale + h));
          } else {
            kd[c] = a[u][0];
            vd[c] = b[u][0];
          }
        }
      }
    }
  }
}

cudaError_t launch_kv_write(const KvWriteParams& p, int num_sms, cudaStream_t stream) {
  if (p.T <= 0) return cudaSuccess;
  const int threads = 256;
  const int warps = threads / 32;
  int blocks = (p.T + warps - 1) / warps;
  const int cap = num_sms * 8;
  if (blocks > cap) blocks = cap;
  size_t smem = p.chunk_lens ? (size_t)(p.B + threads) * sizeof(int32_t) : 0;
  const bool fp8 = p.k_scale != nullptr;
  if (smem > 48 * 1024) {
    cudaError_t e = fp8 ? cudaFuncSetAttribute(kv_write_kernel<true>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)smem)
                        : cudaFuncSetAttribute(kv_write_kernel<false>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)smem);
    if (e != cudaSuccess) return e;
  }
  if (fp8)
    kv_write_kernel<true><<<blocks, threads, smem, stream>>>(p);
  else
    kv_write_kernel<false><<<blocks, threads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
