// pa_combine.cu -- log-sum-exp merge of split-K partial attention states.
//
// Each (sequence, query head) row has S partial states (o_i normalised by its
// own softmax sum, lse_i = natural-log sum of exp(scores) over its keys).
// out = sum_i exp(lse_i - LSE) o_i, LSE = log sum_i exp(lse_i): the softmax
// over the union of the key ranges.  States with lse = -inf hold no keys and
// are skipped (their o is never read, so it may be garbage); any +inf lse
// marks an invalid sequence and zeroes the row.  Memory bound and small: one
// warp per row, each lane owning 4 of the 128 dims (16-byte loads).  Two
// record layouts: fixed splits ([row][split]) and the page-balanced
// schedule's cut units (two records per decode CTA).
#include "pa_launch.cuh"

namespace pa {
namespace {

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__global__ void __launch_bounds__(128) combine_kernel(const CombineParams p) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  // launched as a programmatic dependent of the decode kernel: its partials
  // are complete and visible after this wait
  grid_dependency_wait();
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

__device__ __forceinline__ int bal_pages(int ctx, int max_pages) {
  return (ctx >= 0 && ctx <= max_pages * kPage) ? (ctx + kPage - 1) / kPage : 0;
}

// Page-balanced decode: the decode CTAs form groups of UPS = Hkv * NT (CTA
// g * UPS + j serves unit j, a KV head and token group); the sequences' pages
// laid end to end (n_s pages for sequence s, W in total) are divided among the
// groups, group g taking positions [floor(W g / ng), floor(W (g+1) / ng)).  A
// sequence cut by a group boundary left one partial record per unit in every
// group that touched it: record 2c (CTA c) if the sequence held the group's
// first position, else 2c + 1.  Block b (boundary b = 1 .. ng-1) merges the
// sequence that boundary b cuts, if it starts in group b-1 (so every cut
// sequence is merged exactly once): one warp per output row (new token, query
// head) of the sequence, read from column (t % Lg) G + h % G of unit
// (h / G) NT + t / Lg.
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

__global__ void __launch_bounds__(1024) bal_combine_kernel(const BalCombineParams p) {
  constexpr int kMaxGroups = 1024;
  __shared__ int sh_lo[kMaxGroups + 1];  // group boundaries
  __shared__ int sh_P, sh_s, sh_n, sh_go, sh_W;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int UPS = (p.Hq / p.G) * p.NT;
  const int ng = p.grid / UPS;
  // a boundary's rows (L * Hq) are spread over cpb CTAs, one row per warp
  const int nrows = p.L * p.Hq, wpc = blockDim.x >> 5;
  const int cpb = (nrows + wpc - 1) / wpc;
  const int b = blockIdx.x / cpb + 1, part = blockIdx.x - (b - 1) * cpb;
  if (warp == 0) {
    // prologue, overlapping the decode kernel: locate the sequence at
    // boundary b.  Lane l holds the page counts of sequences 16l .. 16l+15
    // (B <= PA_BALANCED_MAX_SEQS; W < 2^31).
    constexpr int R = PA_BALANCED_MAX_SEQS / 32;
    int np[R];
#pragma unroll
    for (int r = 0; r < R; ++r) np[r] = seq_ctx(p.context_lens, min(lane * R + r, p.B - 1), p.L);
    int lsum = 0;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      np[r] = lane * R + r < p.B ? bal_pages(np[r], p.max_pages) : 0;
      lsum += np[r];
    }
    int incl = lsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const int W = __shfl_sync(0xffffffffu, incl, 31);
    const int X = (int)((int64_t)W * b / ng), lo_prev = (int)((int64_t)W * (b - 1) / ng);
    int start = incl - lsum, hit_r = -1, hit_start = 0;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (hit_r < 0 && np[r] > 0 && start < X && X < start + np[r]) {
        hit_r = r;
        hit_start = start;
      }
      start += np[r];
    }
    const unsigned m = __ballot_sync(0xffffffffu, hit_r >= 0);
    int go = 0, s_hit = 0, n = 0, P = 0;
    if (m) {
      const int f = __ffs(m) - 1;
      const int rr = __shfl_sync(0xffffffffu, hit_r, f);
      s_hit = f * R + rr;
      P = __shfl_sync(0xffffffffu, hit_start, f);
      int nv = 0;
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (r == rr) nv = np[r];
      n = __shfl_sync(0xffffffffu, nv, f);
      go = P >= lo_prev ? 1 : 0;
    }
    if (lane == 0) {
      sh_go = go;
      sh_s = s_hit;
      sh_n = n;
      sh_P = P;
      sh_W = W;
    }
  }
  __syncthreads();
  if (!sh_go) return;
  for (int gg = threadIdx.x; gg <= ng && gg <= kMaxGroups; gg += blockDim.x)
    sh_lo[gg] = (int)((int64_t)sh_W * gg / ng);
  __syncthreads();
  grid_dependency_wait();
  const int P = sh_P, n = sh_n;
  // the groups b-1 .. that touched pages [P, P + n), 32 at a time: lane k
  // holds group b-1+k of the current chunk (its record loads run in parallel)
  for (int r = part * wpc + warp; r < nrows && r < (part + 1) * wpc; r += wpc) {
    const int t = r / p.Hq, hd = r - t * p.Hq;
    const int j = (hd / p.G) * p.NT + t / p.Lg, g = (t % p.Lg) * p.G + hd % p.G;
    float M = -INFINITY;
    bool inval = false;
    for (int g0 = b - 1; g0 < ng; g0 += 32) {
      const int gg = g0 + lane;
      const int lo = gg < ng ? sh_lo[gg] : INT32_MAX, hi = gg < ng ? sh_lo[gg + 1] : INT32_MAX;
      const bool has = gg < ng && lo < P + n && lo != hi;
      const float v = has ? p.bal_lse[(2 * (gg * UPS + j) + (P <= lo ? 0 : 1)) * p.NC + g] : -INFINITY;
      inval |= v == INFINITY;
      M = fmaxf(M, v);
      if (!__any_sync(0xffffffffu, gg < ng && lo < P + n)) break;
    }
    M = warp_max(M);
    inval = __any_sync(0xffffffffu, inval);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!inval && M != -INFINITY) {
      float Lsum = 0.f;
      for (int g0 = b - 1; g0 < ng; g0 += 32) {
        const int gg = g0 + lane;
        const int lo = gg < ng ? sh_lo[gg] : INT32_MAX, hi = gg < ng ? sh_lo[gg + 1] : INT32_MAX;
        const bool has = gg < ng && lo < P + n && lo != hi;
        const int rec = 2 * (gg * UPS + j) + (P <= lo ? 0 : 1);
        const float v = has ? p.bal_lse[rec * p.NC + g] : -INFINITY;
        const float w = v == -INFINITY ? 0.f : expf(v - M);
        Lsum += w;
        unsigned mk = __ballot_sync(0xffffffffu, w != 0.f);
        while (mk) {
          // two records at a time: both loads issue before either is used
          const int k0 = __ffs(mk) - 1;
          mk &= mk - 1;
          const int k1 = mk ? __ffs(mk) - 1 : k0;
          const bool two = mk != 0;
          if (two) mk &= mk - 1;
          const float w0 = __shfl_sync(0xffffffffu, w, k0);
          const float w1 = two ? __shfl_sync(0xffffffffu, w, k1) : 0.f;
          const int r0 = __shfl_sync(0xffffffffu, rec, k0), r1 = __shfl_sync(0xffffffffu, rec, k1);
          const float4 x0 =
              reinterpret_cast<const float4*>(p.bal_o + ((int64_t)r0 * p.NC + g) * kHeadDim)[lane];
          const float4 x1 =
              reinterpret_cast<const float4*>(p.bal_o + ((int64_t)r1 * p.NC + g) * kHeadDim)[lane];
          acc.x = fmaf(w0, x0.x, acc.x);
          acc.y = fmaf(w0, x0.y, acc.y);
          acc.z = fmaf(w0, x0.z, acc.z);
          acc.w = fmaf(w0, x0.w, acc.w);
          if (two) {  // (warp-uniform)
            acc.x = fmaf(w1, x1.x, acc.x);
            acc.y = fmaf(w1, x1.y, acc.y);
            acc.z = fmaf(w1, x1.z, acc.z);
            acc.w = fmaf(w1, x1.w, acc.w);
          }
        }
        if (!__any_sync(0xffffffffu, gg < ng && lo < P + n)) break;
      }
      const float inv = 1.f / warp_sum(Lsum);
      acc = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
    const int64_t row = (int64_t)sh_s * p.L * p.Hq + r;
    if (p.out_f32) {
      reinterpret_cast<float4*>(p.out)[row * (kHeadDim / 4) + lane] = acc;
    } else {
      __nv_bfloat162 a = __floats2bfloat162_rn(acc.x, acc.y);
      __nv_bfloat162 c2 = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&a);
      u.y = *reinterpret_cast<uint32_t*>(&c2);
      reinterpret_cast<uint2*>(p.out)[row * (kHeadDim / 4) + lane] = u;
    }
  }
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  cudaError_t e = launch_dependent(combine_kernel, p, (p.rows + 3) / 4, 128, stream);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

cudaError_t launch_bal_combine(const BalCombineParams& p, cudaStream_t stream) {
  const int ng = p.grid / ((p.Hq / p.G) * p.NT);
  if (ng <= 1) return cudaSuccess;
  // one row per warp: up to 16 warps per CTA, ceil(rows / warps) CTAs per boundary
  const int rows = p.L * p.Hq;
  const int warps = rows < 16 ? rows : 16;
  const int cpb = (rows + warps - 1) / warps;
  cudaError_t e = launch_dependent(bal_combine_kernel, p, (ng - 1) * cpb, 32 * warps, stream);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace pa
