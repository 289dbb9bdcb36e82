// pa_combine.cu -- log-sum-exp merge of split-K partial attention states.
//
// Each (sequence, query head) row has S partial states (o_i normalised by its
// own softmax sum, lse_i = natural-log sum of exp(scores) over its keys).
// out = sum_i exp(lse_i - LSE) o_i, LSE = log sum_i exp(lse_i): the softmax
// over the union of the key ranges.  States with lse = -inf hold no keys and
// are skipped (their o is never read, so it may be garbage); any +inf lse
// marks an invalid sequence and zeroes the row.  Memory bound and small: one
// warp per row, each lane owning 4 of the 128 dims (16-byte loads).
#include "pa_launch.cuh"

namespace pa {
namespace {

__global__ void __launch_bounds__(128) combine_kernel(const CombineParams p) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= p.rows) return;
  const float* lse = p.part_lse + (int64_t)row * p.S;
  float M = -INFINITY;
  bool inval = false;
  for (int i = lane; i < p.S; i += 32) {
    const float v = lse[i];
    inval |= (v == INFINITY);
    M = fmaxf(M, v);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  inval = __any_sync(0xffffffffu, inval);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (!inval && M != -INFINITY) {
    float Lsum = 0.f;
    for (int i = lane; i < p.S; i += 32) {
      const float v = lse[i];
      if (v != -INFINITY) Lsum += expf(v - M);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, o);
    const float inv = 1.f / Lsum;
    const float4* po = reinterpret_cast<const float4*>(p.part_o + (int64_t)row * p.S * kHeadDim);
    for (int i = 0; i < p.S; ++i) {
      const float v = lse[i];
      if (v == -INFINITY) continue;
      const float w = expf(v - M) * inv;
      const float4 x = po[i * (kHeadDim / 4) + lane];
      acc.x = fmaf(w, x.x, acc.x);
      acc.y = fmaf(w, x.y, acc.y);
      acc.z = fmaf(w, x.z, acc.z);
      acc.w = fmaf(w, x.w, acc.w);
    }
  }
  if (p.out_f32) {
    reinterpret_cast<float4*>(p.out)[(int64_t)row * (kHeadDim / 4) + lane] = acc;
  } else {
    __nv_bfloat162 a = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 b = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    reinterpret_cast<uint2*>(p.out)[(int64_t)row * (kHeadDim / 4) + lane] = u;
  }
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  combine_kernel<<<(p.rows + 3) / 4, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
