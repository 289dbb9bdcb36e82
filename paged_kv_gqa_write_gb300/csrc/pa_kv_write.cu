// pa_kv_write.cu -- scatter the new tokens' K/V rows into the paged cache.
//
// "Qwen3-14B" (pypto-lib), "Model structure, top down": the KV cache write
// (decode) / KV cache update (prefill) precedes attention.  "Qwen 3"
// (TensorSharp), section 11: ScatterKv writes each token at slot
// blockId * blockSize + offset.  A pure byte copy, bound by launch latency at
// decode sizes and by HBM at prefill sizes: one warp per token moves the
// token's Hkv*256-byte K row and V row with 16-byte accesses.
#include "pa_launch.cuh"

namespace pa {

__global__ void __launch_bounds__(256) kv_write_kernel(KvWriteParams p) {
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
  for (int token = blockIdx.x * warps_per_block + (threadIdx.x >> 5); token < p.T;
       token += gridDim.x * warps_per_block) {
    int s, j, n;
    if (p.chunk_lens) {
      s = seq_of_token(off, p.B, token);
      if (s >= p.B) continue;  // more tokens than sum(chunk_lens): flagged above
      j = token - (s ? off[s - 1] : 0);
      n = p.chunk_lens[s];
    } else {
      s = token;
      j = 0;
      n = 1;
    }
    const int ctx = p.context_lens[s];
    const int err = warp_check_sequence(p.block_table, s, ctx, n, p.num_pages, p.max_pages);
    if (err) {
      if (lane == 0 && p.status) atomicOr(p.status, err);
      continue;
    }
    const int pos = ctx - n + j;
    const int page = p.block_table[(int64_t)s * p.max_pages + pos / kPage];
    const int64_t slot = (int64_t)page * kPage + pos % kPage;
    const uint4* ks = p.k_new + (int64_t)token * row_chunks;
    const uint4* vs = p.v_new + (int64_t)token * row_chunks;
    uint4* kd = p.k_cache + slot * row_chunks;
    uint4* vd = p.v_cache + slot * row_chunks;
    for (int c = lane; c < row_chunks; c += 32) {
      uint4 a = __ldg(ks + c);
      uint4 b = __ldg(vs + c);
      kd[c] = a;
      vd[c] = b;
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
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kv_write_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kv_write_kernel<<<blocks, threads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
