// pa_topk.cu -- exact top-k of rows of logits (the sampling candidates).
//
// pypto-serving PR #77 ("Qwen3-14B device top-k"), "Exactness Design": an
// exact Top-32 of a row's full-vocabulary logits, merged hierarchically -- the
// union of exact per-group Top-k sets holds the exact global Top-k, because an
// entry outside its group's Top-k has k entries of that group ranked ahead of
// it -- returning the candidate values and token IDs.
//
// Order: larger value first, NaN above +inf, equal values by smaller index
// (-0 and +0 are equal).  Every entry gets a unique 64-bit key: the float's
// bits mapped to an order-preserving integer (NaN to the largest) in the high
// word, the inverted index in the low word; the top k of a set are then the k
// largest keys, with no ties left to break.
//
// Phase 1: a CTA per (row, slice) stages the slice's keys in shared memory
// and finds its k largest by radix select -- one 256-bin histogram pass per
// key byte from the top, each pass restricted to the keys that share the
// digits chosen so far, stopping once the bin holding the k-th key is
// exactly used up -- and writes them as the slice's candidates.  Phase 2 (a
// programmatic dependent launch) runs the same select per row over the
// slices' candidates, sorts the k winners and writes values and indices.  HBM
// bound: each logit is read once.
#include "pa_launch.cuh"

namespace pa {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t order_key(float v) {
  uint32_t u = __float_as_uint(v);
  if (v != v) return 0xFFFFFFFFu;   // NaN ranks above everything
  if (u == 0x80000000u) u = 0u;     // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Selects, among the n keys key_of(i), the k largest (k <= n) into sel[0..k)
// (unordered).  All threads of the block call it; hist and vars are shared.
template <typename F>
__device__ void block_select(int n, int k, F key_of, unsigned long long* sel, int* hist,
                             int* vars /* [4] */) {
  unsigned long long prefix = 0, mask = 0;
  int rem = k;
  for (int sh = 56; sh >= 0; sh -= 8) {
    for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const unsigned long long c = key_of(i);
      if ((c & mask) == prefix) atomicAdd(&hist[(int)((c >> sh) & 255u)], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // the digit v holding the rem-th largest key: lane l sums bins 255-8l .. 248-8l
      const int lane = threadIdx.x;
      int part = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) part += hist[255 - 8 * lane - e];
      int incl = part;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const unsigned m = __ballot_sync(0xffffffffu, incl >= rem);
      const int f = __ffs(m) - 1;  // m != 0: at least rem keys match the prefix
      if (lane == f) {
        int above = incl - part;
        int v = 255 - 8 * lane;
        for (int e = 0; e < 8; ++e, --v) {
          const int h = hist[v];
          if (above + h >= rem) break;
          above += h;
        }
        vars[0] = v;
        vars[1] = above;
        vars[2] = hist[v];
      }
    }
    __syncthreads();
    const int v = vars[0];
    rem -= vars[1];
    prefix |= (unsigned long long)v << sh;
    mask |= 255ull << sh;
    const bool done = vars[2] == rem;  // every key with this prefix is selected
    __syncthreads();                   // vars is rewritten by the next pass
    if (done) break;
  }
  // keys above the prefix, and those equal to it: exactly k
  if (threadIdx.x == 0) vars[3] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const unsigned long long c = key_of(i);
    if ((c & mask) >= prefix) {
      const int pos = atomicAdd(&vars[3], 1);
      if (pos < k) sel[pos] = c;  // exactly k by construction
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads) topk_slice_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint32_t keys[];  // [slice_len]
  __shared__ unsigned long long sel[32];
  __shared__ int hist[256], vars[4];
  const int row = blockIdx.x / p.slices, sl = blockIdx.x - row * p.slices;
  const int lo = sl * p.slice_len;
  const int n = min(p.slice_len, p.vocab - lo);
  const float* src = p.logits + (int64_t)row * p.row_stride + lo;
  // stage the slice's order keys: 16-byte loads from the first 16-byte
  // boundary on, the few entries before it and after the last one by one
  const int head = min(n, (int)(((16u - (uint32_t)(reinterpret_cast<uintptr_t>(src) & 15u)) & 15u) >> 2));
  const int n4 = (n - head) >> 2;
  for (int i = threadIdx.x; i < n4; i += blockDim.x) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(src + head) + i);
    const int b = head + 4 * i;
    keys[b] = order_key(v.x);
    keys[b + 1] = order_key(v.y);
    keys[b + 2] = order_key(v.z);
    keys[b + 3] = order_key(v.w);
  }
  if (threadIdx.x < head) keys[threadIdx.x] = order_key(__ldg(src + threadIdx.x));
  for (int i = head + 4 * n4 + threadIdx.x; i < n; i += blockDim.x) keys[i] = order_key(__ldg(src + i));
  __syncthreads();
  auto key_of = [&](int i) -> unsigned long long {
    return ((unsigned long long)keys[i] << 32) | (uint32_t)~(uint32_t)(lo + i);
  };
  unsigned long long* out = p.cand + ((int64_t)row * p.slices + sl) * p.k;
  if (n <= p.k) {
    // a short slice: all of it (key 0 pads; no entry has key 0)
    for (int j = threadIdx.x; j < p.k; j += blockDim.x) out[j] = j < n ? key_of(j) : 0ull;
    return;
  }
  block_select(n, p.k, key_of, sel, hist, vars);
  for (int j = threadIdx.x; j < p.k; j += blockDim.x) out[j] = sel[j];
}

__global__ void __launch_bounds__(kThreads) topk_merge_kernel(const TopkParams p) {
  extern __shared__ __align__(16) unsigned long long cand[];  // [slices * k]
  __shared__ unsigned long long sel[32];
  __shared__ int hist[256], vars[4];
  const int row = blockIdx.x;
  const int n = p.slices * p.k;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the slice candidates are complete
  const unsigned long long* src = p.cand + (int64_t)row * n;
  for (int i = threadIdx.x; i < n; i += blockDim.x) cand[i] = src[i];
  __syncthreads();
  block_select(n, p.k, [&](int i) { return cand[i]; }, sel, hist, vars);
  if (threadIdx.x < 32) {
    // bitonic sort of the k winners, largest key first (k <= 32; pad with 0)
    const int lane = threadIdx.x;
    unsigned long long x = lane < p.k ? sel[lane] : 0ull;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const unsigned long long y = __shfl_xor_sync(0xffffffffu, x, stride);
        const bool up = (lane & size) == 0;          // this run sorts descending
        const bool lower = (lane & stride) == 0;
        const bool keep_max = (up == lower);
        x = keep_max ? (x > y ? x : y) : (x < y ? x : y);
      }
    }
    if (lane < p.k) {
      const int idx = (int)~(uint32_t)(x & 0xFFFFFFFFull);
      p.out_indices[(int64_t)row * p.k + lane] = idx;
      p.out_values[(int64_t)row * p.k + lane] = __ldg(p.logits + (int64_t)row * p.row_stride + idx);
    }
  }
}

}  // namespace

cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  const size_t smem1 = (size_t)p.slice_len * sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(topk_slice_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
  if (e != cudaSuccess) return e;
  topk_slice_kernel<<<p.rows * p.slices, kThreads, smem1, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem2 = (size_t)p.slices * p.k * sizeof(unsigned long long);
  e = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem2);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.rows);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem2;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, topk_merge_kernel, p);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace pa
