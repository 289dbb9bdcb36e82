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
// Phase 1: a CTA per (row, slice) stages the slice's keys in shared memory,
// tracking each thread's largest.  Each warp offers its ceil(k / warps)-th
// largest lane maximum; the smallest offer is a threshold that at least k keys
// reach (that many distinct lanes of every warp hold one), and for any but
// contrived data few keys more: the keys at or above it are gathered, ranked
// against each other, and the k best written in order as the slice's
// candidates.  When too many keys reach the threshold, a radix select over
// the whole slice takes over (one 256-bin histogram pass per key
// byte from the top, stopping once the bin holding the k-th key is exactly
// used up).  Phase 2 (a programmatic dependent launch) is a warp per row that
// folds the slices' sorted candidate lists into one sorted top-k, a bitonic
// merge per list.  HBM bound: each logit is read once.
#include "pa_launch.cuh"

namespace pa {
namespace {

constexpr int kThreads = 256;  // a multiple of 32

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

constexpr int kCap = 1024;  // gathered keys ranked directly; more take the radix select

// Writes the k largest of the n keys key_of(i) (all distinct), larger first,
// to out[0..k): each key's rank is the number of keys above it.  Keys past n
// are written as 0 (below every key).  All threads of the block call it.
template <typename F>
__device__ void block_rank_write(int n, int k, F key_of, unsigned long long* out) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const unsigned long long c = key_of(i);
    int r = 0;
    for (int j = 0; j < n; ++j) r += key_of(j) > c ? 1 : 0;
    if (r < k) out[r] = c;
  }
  for (int j = n + threadIdx.x; j < k; j += blockDim.x) out[j] = 0ull;
}

__global__ void __launch_bounds__(kThreads) topk_slice_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint32_t keys[];  // [slice_len]
  __shared__ unsigned long long sel[32];
  __shared__ unsigned long long gath[kCap];
  __shared__ int hist[256], vars[4];
  __shared__ uint32_t thr;
  __shared__ int ngath;
  // the merge grid may start now: it waits for this grid's results
  asm volatile("griddepcontrol.launch_dependents;");
  const int row = blockIdx.x / p.slices, sl = blockIdx.x - row * p.slices;
  const int lo = sl * p.slice_len;
  const int n = min(p.slice_len, p.vocab - lo);
  const float* src = p.logits + (int64_t)row * p.row_stride + lo;
  // stage the slice's order keys: 16-byte loads from the first 16-byte
  // boundary on, the few entries before it and after the last one by one;
  // each thread keeps the largest key it staged
  const int head = min(n, (int)(((16u - (uint32_t)(reinterpret_cast<uintptr_t>(src) & 15u)) & 15u) >> 2));
  const int n4 = (n - head) >> 2;
  uint32_t mx = 0;  // below every key
  constexpr int kBatch = 8;  // 16-byte loads in flight per thread
  for (int i0 = threadIdx.x; i0 < n4; i0 += kBatch * kThreads) {
    float4 v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = i0 + u * kThreads;
      if (i < n4) v[u] = __ldg(reinterpret_cast<const float4*>(src + head) + i);
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = i0 + u * kThreads;
      if (i < n4) {
        const int b = head + 4 * i;
        const uint32_t k0 = order_key(v[u].x), k1 = order_key(v[u].y), k2 = order_key(v[u].z),
                       k3 = order_key(v[u].w);
        keys[b] = k0;
        keys[b + 1] = k1;
        keys[b + 2] = k2;
        keys[b + 3] = k3;
        mx = max(mx, max(max(k0, k1), max(k2, k3)));
      }
    }
  }
  if (threadIdx.x < head) {
    const uint32_t k0 = order_key(__ldg(src + threadIdx.x));
    keys[threadIdx.x] = k0;
    mx = max(mx, k0);
  }
  for (int i = head + 4 * n4 + threadIdx.x; i < n; i += blockDim.x) {
    const uint32_t k0 = order_key(__ldg(src + i));
    keys[i] = k0;
    mx = max(mx, k0);
  }
  if (threadIdx.x == 0) {
    ngath = 0;
    thr = 0xFFFFFFFFu;
  }
  __syncthreads();
  // the threshold: each warp sorts its lanes' maxima (bitonic, larger first)
  // and offers its ceil(k / warps)-th largest; the smallest offer is reached
  // by at least that many keys in every warp, so by at least k keys
  {
    const int lane = threadIdx.x & 31;
    uint32_t x = mx;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const uint32_t y = __shfl_xor_sync(0xffffffffu, x, stride);
        const bool keep_max = ((lane & size) == 0) == ((lane & stride) == 0);
        x = keep_max ? max(x, y) : min(x, y);
      }
    }
    const int per = (p.k + kThreads / 32 - 1) / (kThreads / 32);
    const uint32_t offer = __shfl_sync(0xffffffffu, x, per - 1);
    if (lane == 0) atomicMin(&thr, offer);  // offer 0 (lanes without keys): gather all
  }
  __syncthreads();
  auto key_of = [&](int i) -> unsigned long long {
    return ((unsigned long long)keys[i] << 32) | (uint32_t)~(uint32_t)(lo + i);
  };
  unsigned long long* out = p.cand + ((int64_t)row * p.slices + sl) * p.k;
  const uint32_t t = thr;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    if (keys[i] >= t) {
      const int pos = atomicAdd(&ngath, 1);
      if (pos < kCap) gath[pos] = key_of(i);
    }
  }
  __syncthreads();
  const int c = ngath;  // >= min(k, n)
  if (c <= kCap) {
    block_rank_write(c, p.k, [&](int i) { return gath[i]; }, out);
    return;
  }
  // many keys at the threshold (heavy ties): radix select over the slice,
  // then rank the k selected
  block_select(n, p.k, key_of, sel, hist, vars);
  block_rank_write(p.k, p.k, [&](int i) { return sel[i]; }, out);
}

// One warp per row: the slices' candidate lists, each sorted (larger first,
// 0 = none), folded into the row's top k.
__global__ void __launch_bounds__(32) topk_merge_kernel(const TopkParams p) {
  const int row = blockIdx.x, lane = threadIdx.x;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the slice candidates are complete
  const unsigned long long* src = p.cand + (int64_t)row * p.slices * p.k;
  unsigned long long cur = lane < p.k ? src[lane] : 0ull;  // sorted across lanes, larger first
  constexpr int kAhead = 8;
  for (int s0 = 1; s0 < p.slices; s0 += kAhead) {
    unsigned long long nx[kAhead];
#pragma unroll
    for (int u = 0; u < kAhead; ++u)
      nx[u] = (s0 + u < p.slices && lane < p.k) ? src[(int64_t)(s0 + u) * p.k + lane] : 0ull;
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      if (s0 + u >= p.slices) break;
      // the top 32 of two sorted lists: element-wise max against the other
      // list reversed (a bitonic sequence), then a bitonic clean
      const unsigned long long b = __shfl_sync(0xffffffffu, nx[u], 31 - lane);
      unsigned long long x = cur > b ? cur : b;
#pragma unroll
      for (int stride = 16; stride > 0; stride >>= 1) {
        const unsigned long long y = __shfl_xor_sync(0xffffffffu, x, stride);
        x = (lane & stride) ? (x < y ? x : y) : (x > y ? x : y);
      }
      cur = x;
    }
  }
  if (lane < p.k) {
    const int idx = (int)~(uint32_t)(cur & 0xFFFFFFFFull);
    p.out_indices[(int64_t)row * p.k + lane] = idx;
    p.out_values[(int64_t)row * p.k + lane] = __ldg(p.logits + (int64_t)row * p.row_stride + idx);
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.rows);
  cfg.blockDim = dim3(32);
  cfg.dynamicSmemBytes = 0;
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
