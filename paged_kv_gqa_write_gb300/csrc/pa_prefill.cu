// pa_prefill.cu -- causal chunked-prefill attention over the paged cache on
// the 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// "Qwen3-14B" (pypto-lib), "prefill_fwd": per layer the KV cache update is
// followed by causal attention over token-major packed inputs
// (T = sum(chunk_lens)).  "Qwen 3" (TensorSharp), 4.1 "Attention": full
// causal GQA, no window or sinks.  New token j of sequence s sits at
// position ctx[s] - chunk_lens[s] + j and attends to keys 0..position of its
// own sequence, read from the paged cache (prior context plus the chunk,
// which pa_kv_write has already stored).
//
// Work item: (sequence, 128-token query tile, query head).  S = Q K^T and
// O += P V are dense 128x128x128 BF16 products per 128-token key page.
//  * warp 0, one lane: TMA producer -- the Q tile (3-D map over [T, Hq, 128])
//    and a 2-deep ring each of K and V page tiles (128-byte swizzle), in the
//    layout the tensor core reads directly.
//  * warp 1, one lane: issues tcgen05.mma (M=128, N=128, K=16 steps) for
//    S_j = Q K_j^T into one of two TMEM score buffers, then O += P_{j-1} V_{j-1}
//    with V as an MN-major operand, committing completions to mbarriers.  The
//    warp also owns the TMEM allocation (512 columns: S0, S1, O).
//  * warps 2-5: one thread per query row.  tcgen05.ld of the score row,
//    causal mask (only on tiles that cross the row's position), online
//    softmax in the log2 domain; P (BF16) goes to a swizzled shared-memory
//    tile the next MMA reads.  O is rescaled in TMEM only when the running
//    max grows by more than 2^8 (the final O / l is unchanged by the choice of
//    reference max).  The epilogue divides by l and writes the row.
// Key pages entirely above the tile's last query position are never loaded
// (causal tile skipping); V rows past the sequence's context in its last page
// are zeroed in shared memory before use (P is 0 there, but 0 * NaN is NaN).
#include "pa_launch.cuh"

namespace pa {
namespace {

constexpr int kThreads = 192;
constexpr int kTileBytes = 128 * 128 * 2;     // 32 KB: one 128x128 bf16 tile
constexpr int kBox = 16384;                   // 64-column half of a tile
constexpr int kRing = 2;
// shared memory layout (offsets from a 1024-aligned base)
constexpr int kQ = 0;
constexpr int kK = kQ + kTileBytes;
constexpr int kV = kK + kRing * kTileBytes;
constexpr int kP = kV + kRing * kTileBytes;
constexpr int kBars = kP + kRing * kTileBytes;
constexpr int kNumBars = 2 + 4 * kRing + 4 * 2 + 2;
constexpr int kSmem = kBars + kNumBars * 8 + 16 + 1024;
// TMEM columns
constexpr uint32_t kColS = 0;     // two 128-column score buffers
constexpr uint32_t kColO = 256;   // 128-column output accumulator
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct Bars {
  uint64_t* q_full;
  uint64_t* q_empty;
  uint64_t* k_full;   // [kRing]
  uint64_t* k_empty;
  uint64_t* v_full;
  uint64_t* v_empty;
  uint64_t* s_full;   // [2]
  uint64_t* s_free;
  uint64_t* p_full;
  uint64_t* p_free;
  uint64_t* o_done;
  uint64_t* o_free;
};

// Walks (sequence, query tile, head) items in increasing order.
struct Cursor {
  int s = 0, tiles_before = 0, tok_before = 0;
  __device__ __forceinline__ int tiles_of(const PrefillParams& p, int seq) const {
    const int n = __ldg(p.chunk_lens + seq);
    return n > 0 ? (n + 127) / 128 : 0;
  }
  // Advance to the sequence holding query tile `tile`; false when past the end.
  __device__ __forceinline__ bool seek(const PrefillParams& p, int tile) {
    while (s < p.B) {
      const int nt = tiles_of(p, s);
      if (tile < tiles_before + nt) return true;
      tiles_before += nt;
      const int n = __ldg(p.chunk_lens + s);
      tok_before += n > 0 ? n : 0;
      ++s;
    }
    return false;
  }
};

struct Item {
  int s, g, h, qt;
  int tok0;      // packed index of the tile's first query token
  int nrows;     // query rows of this tile that exist (<= 128)
  int prior;     // context before the chunk
  int ctx;
  int nkt;       // key tiles to visit (0: lengths invalid)
  bool len_ok;
};

__device__ __forceinline__ Item make_item(const PrefillParams& p, const Cursor& c, int tile,
                                          int g) {
  Item it;
  it.s = c.s;
  it.g = g;
  it.h = g / p.G;
  it.qt = tile - c.tiles_before;
  const int n = __ldg(p.chunk_lens + c.s);
  it.ctx = __ldg(p.context_lens + c.s);
  it.tok0 = c.tok_before + it.qt * 128;
  it.nrows = min(128, n - it.qt * 128);
  it.len_ok = it.ctx >= 0 && n >= 0 && n <= it.ctx && it.ctx <= p.max_pages * kPage;
  it.prior = it.ctx - n;
  it.nkt = it.len_ok ? (it.prior + it.qt * 128 + it.nrows - 1) / kPage + 1 : 0;
  return it;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_q, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kBars);
  Bars B;
  B.q_full = bar;
  B.q_empty = bar + 1;
  B.k_full = bar + 2;
  B.k_empty = B.k_full + kRing;
  B.v_full = B.k_empty + kRing;
  B.v_empty = B.v_full + kRing;
  B.s_full = B.v_empty + kRing;
  B.s_free = B.s_full + 2;
  B.p_full = B.s_free + 2;
  B.p_free = B.p_full + 2;
  B.o_done = B.p_free + 2;
  B.o_free = B.o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBars + kNumBars * 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(B.q_full, 1);
    mbar_init(B.q_empty, 1);
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&B.k_full[i], 1);
      mbar_init(&B.k_empty[i], 1);
      mbar_init(&B.v_full[i], 1);
      mbar_init(&B.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B.s_full[i], 1);
      mbar_init(&B.s_free[i], 128);
      mbar_init(&B.p_full[i], 128);
      mbar_init(&B.p_free[i], 1);
    }
    mbar_init(B.o_done, 1);
    mbar_init(B.o_free, 128);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensor_map(&tm_q);
      prefetch_tensor_map(&tm_k);
      prefetch_tensor_map(&tm_v);
      const uint64_t pol_kv = l2_policy_evict_last();  // reused by other tiles/heads
      const uint64_t pol_q = l2_policy_evict_first();
      Cursor cur;
      uint32_t items = 0, tiles = 0;
      bool ok = true;
      for (int i = blockIdx.x; ok; i += gridDim.x) {
        const int tile = i / p.Hq, g = i - tile * p.Hq;
        if (!cur.seek(p, tile)) break;
        const Item it = make_item(p, cur, tile, g);
        if (it.nkt == 0) continue;
        ok = mbar_wait(B.q_empty, (items & 1) ^ 1, p.status);
        if (!ok) break;
        mbar_arrive_expect_tx(B.q_full, kTileBytes);
        tma_load_3d(smem + kQ, &tm_q, 0, it.g, it.tok0, B.q_full, pol_q);
        tma_load_3d(smem + kQ + kBox, &tm_q, 64, it.g, it.tok0, B.q_full, pol_q);
        ++items;
        const int32_t* bt = p.block_table + (int64_t)it.s * p.max_pages;
        for (int kt = 0; kt < it.nkt; ++kt, ++tiles) {
          int page = __ldg(bt + kt);
          if (page < 0 || page >= p.num_pages) page = 0;  // sequence reported invalid
          const int slot = tiles % kRing;
          const uint32_t ph = ((tiles / kRing) & 1) ^ 1;
          const int x = it.h * kHeadDim, y = page * kPage;
          if (!(ok = mbar_wait(&B.k_empty[slot], ph, p.status))) break;
          mbar_arrive_expect_tx(&B.k_full[slot], kTileBytes);
          tma_load_2d(smem + kK + slot * kTileBytes, &tm_k, x, y, &B.k_full[slot], pol_kv);
          tma_load_2d(smem + kK + slot * kTileBytes + kBox, &tm_k, x + 64, y, &B.k_full[slot],
                      pol_kv);
          if (!(ok = mbar_wait(&B.v_empty[slot], ph, p.status))) break;
          mbar_arrive_expect_tx(&B.v_full[slot], kTileBytes);
          tma_load_2d(smem + kV + slot * kTileBytes, &tm_v, x, y, &B.v_full[slot], pol_kv);
          tma_load_2d(smem + kV + slot * kTileBytes + kBox, &tm_v, x + 64, y, &B.v_full[slot],
                      pol_kv);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = umma_idesc_bf16(128, 128, false, false);
      const uint32_t idesc_pv = umma_idesc_bf16(128, 128, false, true);
      const uint32_t q_addr = smem_u32(smem + kQ);
      Cursor cur;
      uint32_t items = 0, tiles = 0;
      bool ok = true;
      // P.V for global tile index j (its P buffer j%2, its V ring slot j%kRing)
      auto issue_pv = [&](uint32_t j, bool first_of_item) -> bool {
        const int pb = j & 1, vs = j % kRing;
        if (!mbar_wait(&B.p_full[pb], (j >> 1) & 1, p.status)) return false;
        if (!mbar_wait(&B.v_full[vs], (j / kRing) & 1, p.status)) return false;
        if (first_of_item && items > 1 && !mbar_wait(B.o_free, (items & 1), p.status))
          return false;
        tc_fence_after();
        const uint32_t p_addr = smem_u32(smem + kP + pb * kTileBytes);
        const uint32_t v_addr = smem_u32(smem + kV + vs * kTileBytes);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t ad = umma_sdesc_sw128(p_addr + (k >> 2) * kBox + (k & 3) * 32, 16, 1024);
          const uint64_t bd = umma_sdesc_sw128(v_addr + k * 2048, kBox, 1024);
          umma_bf16_ss(tmem + kColO, ad, bd, idesc_pv, (first_of_item && k == 0) ? 0u : 1u);
        }
        umma_commit(&B.v_empty[vs]);
        umma_commit(&B.p_free[pb]);
        umma_commit(B.o_done);
        return true;
      };
      for (int i = blockIdx.x; ok; i += gridDim.x) {
        const int tile = i / p.Hq, g = i - tile * p.Hq;
        if (!cur.seek(p, tile)) break;
        const Item it = make_item(p, cur, tile, g);
        if (it.nkt == 0) continue;
        if (!(ok = mbar_wait(B.q_full, items & 1, p.status))) break;
        ++items;
        const uint32_t first = tiles;
        for (int kt = 0; kt < it.nkt; ++kt, ++tiles) {
          const int ks = tiles % kRing, sb = tiles & 1;
          if (!(ok = mbar_wait(&B.k_full[ks], (tiles / kRing) & 1, p.status))) break;
          if (!(ok = mbar_wait(&B.s_free[sb], ((tiles >> 1) & 1) ^ 1, p.status))) break;
          tc_fence_after();
          const uint32_t k_addr = smem_u32(smem + kK + ks * kTileBytes);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint64_t ad = umma_sdesc_sw128(q_addr + (k >> 2) * kBox + (k & 3) * 32, 16, 1024);
            const uint64_t bd = umma_sdesc_sw128(k_addr + (k >> 2) * kBox + (k & 3) * 32, 16, 1024);
            umma_bf16_ss(tmem + kColS + sb * 128, ad, bd, idesc_qk, k > 0 ? 1u : 0u);
          }
          umma_commit(&B.s_full[sb]);
          umma_commit(&B.k_empty[ks]);
          if (kt == it.nkt - 1) umma_commit(B.q_empty);
          if (kt > 0 && !(ok = issue_pv(tiles - 1, tiles - 1 == first))) break;
        }
        if (!ok) break;
        if (!(ok = issue_pv(tiles - 1, tiles - 1 == first))) break;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const int quarter = warp & 3;            // TMEM lanes this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int t = threadIdx.x - 64;          // 0..127 among softmax threads
    if (blockIdx.x == 0 && warp == 2 && p.status) {
      int sum = 0;
      for (int e = lane; e < p.B; e += 32) sum += max(__ldg(p.chunk_lens + e), 0);
#pragma unroll
      for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (lane == 0 && sum != p.T) atomicOr(p.status, PA_STATUS_BAD_TOKENS);
    }
    Cursor cur;
    uint32_t items = 0, tiles = 0;
    bool ok = true;
    for (int i = blockIdx.x; ok; i += gridDim.x) {
      const int tile = i / p.Hq, g = i - tile * p.Hq;
      if (!cur.seek(p, tile)) break;
      const Item it = make_item(p, cur, tile, g);
      // sequence validity: lengths and every referenced block-table entry
      bool bad = !it.len_ok;
      if (!bad) {
        const int used = (it.ctx + kPage - 1) / kPage;
        const int32_t* bt = p.block_table + (int64_t)it.s * p.max_pages;
        bool b = false;
        for (int e = lane; e < used; e += 32) {
          const int pg = __ldg(bt + e);
          b |= (pg < 0 || pg >= p.num_pages);
        }
        bad = __any_sync(0xffffffffu, b);
      }
      if (bad && t == 0 && it.qt == 0 && g == 0 && p.status)
        atomicOr(p.status, it.len_ok ? PA_STATUS_BAD_PAGE : PA_STATUS_BAD_LENGTH);
      const int64_t tok = (int64_t)it.tok0 + row;
      const bool row_out = row < it.nrows && tok < p.T;
      if (it.nkt == 0) {
        if (row_out) {
          uint8_t* dst = reinterpret_cast<uint8_t*>(p.out) +
                         ((tok * p.Hq + it.g) * kHeadDim) * (p.out_f32 ? 4 : 2);
          for (int c = 0; c < (p.out_f32 ? 32 : 16); ++c)
            reinterpret_cast<uint4*>(dst)[c] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      ++items;
      const int pos = it.prior + it.qt * 128 + min(row, it.nrows - 1);  // query position
      const int last_page = (it.ctx - 1) / kPage;
      const int vtail = it.ctx % kPage;  // rows >= vtail of the last page are past the context
      float m = -INFINITY, l = 0.f;
      uint32_t first = tiles;
      for (int kt = 0; kt < it.nkt; ++kt, ++tiles) {
        const int sb = tiles & 1;
        if (!(ok = mbar_wait_warp(&B.s_full[sb], (tiles >> 1) & 1, p.status))) break;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_base + kColS + sb * 128 + c * 32, sr[c]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&B.s_free[sb]);
        // scores in log2 units, causal mask only where the tile crosses pos
        const int key0 = kt * kPage;
        const bool full = key0 + kPage - 1 <= pos;
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            float x = __uint_as_float(sr[c][e]) * p.scale_log2;
            if (!full && key0 + c * 32 + e > pos) x = -INFINITY;
            sr[c][e] = __float_as_uint(x);
            mx = fmaxf(mx, x);
          }
        const float m_new = fmaxf(m, mx);
        bool rescale = false;
        float alpha = 1.f;
        if (m == -INFINITY) {
          m = m_new;
        } else if (m_new > m + kRescaleThreshold) {
          alpha = fast_exp2(m - m_new);
          rescale = true;
          m = m_new;
        }
        // P buffer sb is free once the P.V two tiles back has completed
        if (!(ok = mbar_wait_warp(&B.p_free[sb], ((tiles >> 1) & 1) ^ 1, p.status))) break;
        const uint32_t pbase = smem_u32(smem + kP + sb * kTileBytes) + row * 128;
        float sum = 0.f;
#pragma unroll
        for (int ch = 0; ch < 16; ++ch) {  // 8 keys per 16-byte chunk
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int k0 = ch * 8 + 2 * e;
            const float p0 = fast_exp2(__uint_as_float(sr[k0 >> 5][k0 & 31]) - m);
            const float p1 = fast_exp2(__uint_as_float(sr[(k0 + 1) >> 5][(k0 + 1) & 31]) - m);
            sum += p0 + p1;
            w[e] = pack_bf16x2(p0, p1);
          }
          sts128(pbase + (ch >> 3) * kBox + (((ch & 7) ^ (row & 7)) << 4), w[0], w[1], w[2], w[3]);
        }
        l = l * alpha + sum;
        if (kt == it.nkt - 1 && kt == last_page && vtail != 0) {
          // zero V rows past the context in the last page before P.V reads them
          const int vs = tiles % kRing;
          if (!(ok = mbar_wait_warp(&B.v_full[vs], (tiles / kRing) & 1, p.status))) break;
          const int r = vtail + t;
          if (r < kPage) {
            const uint32_t vb = smem_u32(smem + kV + vs * kTileBytes) + r * 128;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
              sts128(vb + ch * 16, 0u, 0u, 0u, 0u);
              sts128(vb + kBox + ch * 16, 0u, 0u, 0u, 0u);
            }
          }
        }
        fence_proxy_async_smem();
        if (rescale && tiles > first) {
          // O holds P.V up to the previous tile: wait for it, then scale in place
          if (!(ok = mbar_wait_warp(B.o_done, (tiles - 1) & 1, p.status))) break;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t orow[32];
            tmem_ld32(tmem + lane_base + kColO + c * 32, orow);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) orow[e] = __float_as_uint(__uint_as_float(orow[e]) * alpha);
            tmem_st32(tmem + lane_base + kColO + c * 32, orow);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(&B.p_full[sb]);
      }
      if (!ok) break;
      // ---- epilogue: O / l for this row
      if (!(ok = mbar_wait_warp(B.o_done, (tiles - 1) & 1, p.status))) break;
      tc_fence_after();
      const float inv = l == 0.f ? 0.f : 1.f / l;
      // an invalid sequence may have read a substitute page: select zeros
      const uint32_t keep = bad ? 0u : 0xffffffffu;
      uint8_t* dst = reinterpret_cast<uint8_t*>(p.out) +
                     ((tok * p.Hq + it.g) * kHeadDim) * (p.out_f32 ? 4 : 2);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t orow[32];
        tmem_ld32(tmem + lane_base + kColO + c * 32, orow);
        tmem_wait_ld();
        if (row_out) {
          if (p.out_f32) {
            uint4* d4 = reinterpret_cast<uint4*>(dst) + c * 8;
#pragma unroll
            for (int e = 0; e < 8; ++e)
              d4[e] = make_uint4(__float_as_uint(__uint_as_float(orow[4 * e]) * inv) & keep,
                                 __float_as_uint(__uint_as_float(orow[4 * e + 1]) * inv) & keep,
                                 __float_as_uint(__uint_as_float(orow[4 * e + 2]) * inv) & keep,
                                 __float_as_uint(__uint_as_float(orow[4 * e + 3]) * inv) & keep);
          } else {
            uint4* d4 = reinterpret_cast<uint4*>(dst) + c * 4;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float* f = reinterpret_cast<const float*>(orow) + 8 * e;
              d4[e] = make_uint4(pack_bf16x2(f[0] * inv, f[1] * inv) & keep,
                                 pack_bf16x2(f[2] * inv, f[3] * inv) & keep,
                                 pack_bf16x2(f[4] * inv, f[5] * inv) & keep,
                                 pack_bf16x2(f[6] * inv, f[7] * inv) & keep);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(B.o_free);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                           const CUtensorMap& tm_q, const PrefillParams& p, int num_sms,
                           cudaStream_t stream) {
  static_assert(kSmem <= 232448, "prefill shared memory exceeds the per-CTA limit");
  cudaError_t e =
      cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM (tensor memory and shared memory are sized for one)
  const int64_t max_items = ((int64_t)p.T / 128 + p.B) * p.Hq;
  const int grid = (int)(max_items < num_sms ? max_items : num_sms);
  if (grid < 1) return cudaSuccess;
  prefill_kernel<<<grid, kThreads, kSmem, stream>>>(tm_k, tm_v, tm_q, p);
  return cudaGetLastError();
}

}  // namespace pa
