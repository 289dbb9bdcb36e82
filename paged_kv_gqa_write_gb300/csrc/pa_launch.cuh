// pa_launch.cuh -- kernel launchers, one per translation unit, called by the C ABI layer.
#pragma once
#include "pa_common.cuh"

namespace pa {

// Launch as a programmatic dependent of the kernel before it on the stream
// (its prologue may overlap that kernel; griddepcontrol.wait orders the reads).
template <typename P>
inline cudaError_t launch_dependent(void (*kernel)(P), const P& p, int grid, int block,
                             cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}


cudaError_t launch_kv_write(const KvWriteParams& p, int num_sms, cudaStream_t stream);

// Q/K RMSNorm, NeoX RoPE and the KV write of the new tokens, fused.
cudaError_t launch_prologue(const PrologueParams& p, int num_sms, cudaStream_t stream);

// Decode: persistent flash-decoding kernel over (split, sequence, kv head,
// token group) items.  tm_k / tm_v are 2-D tensor maps over the caches viewed
// as [num_pages * 128 rows, Hkv * 128 columns] bf16 with 128-byte swizzle and
// a 64 x 128 box; tm_q is a 2-D map over q viewed as [B * Hq rows, 128
// columns] with a 64 x gc box (gc = query heads per item, <= 16).
// With p.k_scale set the caches are e4m3 (uint8 maps, 128 x 128 boxes); with
// p.L > 1, tm_q is a 3-D map over [tokens][Hq][128] with a 64 x G x Lg box.
cudaError_t launch_decode(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                          const CUtensorMap& tm_q, const DecodeParams& p, int gc, int num_sms,
                          cudaStream_t stream);

// Decode with its prologue in the kernel (bf16 cache, one token per sequence,
// g = Hq / Hkv <= 16): q is built from pro.qkv, the new tokens' K/V rows are
// written to pro.k_cache / pro.v_cache; no q tensor map.
cudaError_t launch_decode_prologue(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                   const DecodeParams& p, const DecodePrologue& pro, int g,
                                   int num_sms, cudaStream_t stream);

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream);

// Merge of the units a page-balanced decode launch of p.grid CTAs cut.
cudaError_t launch_bal_combine(const BalCombineParams& p, cudaStream_t stream);

// Exact top-k of logit rows: per-slice candidates, then a per-row merge.
cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream);

// One CTA whose waiting warp waits, with the kernels' bounded wait, on an
// mbarrier that nothing arrives on, giving up after limit_ns.
cudaError_t launch_wait_selftest(uint64_t limit_ns, int32_t* status, cudaStream_t stream);

// CTA pairs a prefill launch uses at most on the current device (the pairs
// that can be resident at once), cached per device.
cudaError_t prefill_pairs(int num_sms, int* pairs);

// tm_o: 3-D map over a BF16 out [T][Hq][128] with 64 x 1 x 128 boxes and
// 128-byte swizzle (unused, any contents, for FP32 output).  p.k_scale
// non-null selects the FP8-cache kernel: tm_k and tm_v are then maps over the
// e4m3 caches, K with 128-byte x 64-row boxes (128-byte swizzle) and V with
// 64-byte x 128-row boxes (64-byte swizzle).
cudaError_t launch_prefill(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                           const CUtensorMap& tm_q, const CUtensorMap& tm_o,
                           const PrefillParams& p, int num_sms, cudaStream_t stream);

}  // namespace pa
