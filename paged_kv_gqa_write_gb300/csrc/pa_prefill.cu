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
// Work item: (sequence, pair of consecutive 128-token query tiles A and B,
// query head).  Both tiles share every K/V page tile the CTA loads, so each
// 64 KB of K/V feeds four 128x128x128 BF16 products (S_A, S_B, P_A.V, P_B.V):
// with one query tile per load the kernel would be bound by L2 bandwidth
// (~72 GB/s per SM), with two it needs half that.
//  * warp 0 (one lane) loads the two Q tiles (3-D TMA map over [T, Hq, 128])
//    and the K page tiles into a 3-deep ring; warp 10 (one lane) the V page
//    tiles into a 2-deep ring (128-byte swizzle, the layout the tensor core
//    reads).
//  * warp 1 (one lane) issues tcgen05.mma (M=128, N=128, K=16 steps) in the
//    order P_A(j).V(j), S_A(j+1), P_B(j).V(j), S_B(j+1), so that each softmax
//    group overlaps the other's MMAs.  P_t(j) is read from tensor memory (it
//    overwrites the first 64 columns of S_t(j) as packed BF16 pairs); V is an
//    MN-major shared-memory operand.  The MMAs of one thread execute in issue
//    order, so P_t(j) is consumed before S_t(j+1) is written.  The warp owns
//    the TMEM allocation (S_A, S_B, O_A, O_B: 512 columns).
//  * warps 2-5 (tile A) and 6-9 (tile B): one thread per query row.  Per key
//    tile: tcgen05.ld of the score row, causal mask (only on tiles that cross
//    the row's position), online softmax in the log2 domain (max of the raw
//    scores, one FMA + exp2 per element), P into TMEM.  O_t is rescaled in
//    TMEM only when the max grows by more than 2^8 (the final O / l is
//    unchanged by the choice of reference max).  Epilogue: O_t / l per row.
// Key pages entirely above a tile's last query position are never loaded for
// it (causal tile skipping); V rows past the sequence's context in its last
// page are zeroed in shared memory before use (P is 0 there, but 0 * NaN is
// NaN).  Items are dealt to the persistent CTAs in decreasing order of
// key-tile count, snaking across CTAs (a greedy longest-first balance every
// CTA computes from the lengths); very large launches fall back to
// round-robin.
#include <type_traits>

#include "pa_launch.cuh"

namespace pa {
namespace {

constexpr int kVWarp = 10;                    // V producer
constexpr int kThreads = (kVWarp + 1) * 32;
constexpr int kTileBytes = 128 * 128 * 2;     // 32 KB: one 128x128 bf16 tile
constexpr int kBox = 16384;                   // 64-column half of a tile
constexpr int kRingK = 2, kRingV = 3;
constexpr int kMaxList = 64;                  // scheduled items per CTA
// shared memory layout (offsets from a 1024-aligned base)
constexpr int kQ = 0;                         // Q_A, Q_B
constexpr int kK = kQ + 2 * kTileBytes;
constexpr int kV = kK + kRingK * kTileBytes;
constexpr int kListInts = 5;                  // per item: s, pair|head, tok0, chunk len, ctx
constexpr int kList = kV + kRingV * kTileBytes;  // schedule [kMaxList][kListInts] int
constexpr int kBars = kList + kMaxList * kListInts * 4;
constexpr int kNumBars = 2 * 2 + 2 * kRingK + 2 * kRingV + 4 * 2;
constexpr int kSmem = kBars + kNumBars * 8 + 16 + 1024;
constexpr int kMaxCost = 4096;                // schedule histogram buckets (ring scratch)
constexpr int kMaxSchedSeqs = (kRingV * kTileBytes / 4 - 1) / 4;  // sequences the schedule stages
// TMEM columns
constexpr uint32_t kColS = 0;     // S_A, S_B: 128 columns each (P in their first 64)
constexpr uint32_t kColO = 256;   // O_A, O_B: 128 columns each
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct Bars {
  uint64_t* q_full;   // [2] per query tile
  uint64_t* q_empty;
  uint64_t* k_full;   // [kRingK]
  uint64_t* k_empty;
  uint64_t* v_full;   // [kRingV]
  uint64_t* v_empty;
  uint64_t* s_full;   // [2] per query tile
  uint64_t* p_full;
  uint64_t* o_done;
  uint64_t* o_free;
};

struct Item {
  int s, g, h, pair;
  int tok0;          // packed index of tile A's first query token
  int nrows[2];      // query rows of tiles A, B (<= 128; B may be 0)
  int nkt[2];        // key tiles each query tile visits (0: none / lengths invalid)
  int nmax;          // key tiles the pair loads
  int prior, ctx;
  bool len_ok;
};

__device__ __forceinline__ bool lengths_ok(const PrefillParams& p, int n, int ctx) {
  return ctx >= 0 && n >= 0 && n <= ctx && ctx <= p.max_pages * kPage;
}

__device__ __forceinline__ Item make_item(const PrefillParams& p, int s, int pair, int g,
                                          int tok0, int n, int ctx) {
  Item it;
  it.s = s;
  it.g = g;
  it.h = g / p.G;
  it.pair = pair;
  it.ctx = ctx;
  it.tok0 = tok0;
  it.len_ok = lengths_ok(p, n, it.ctx);
  it.prior = it.ctx - n;
  for (int t = 0; t < 2; ++t) {
    const int q0 = pair * 256 + t * 128;
    it.nrows[t] = max(0, min(128, n - q0));
    it.nkt[t] = (it.len_ok && it.nrows[t] > 0) ? (it.prior + q0 + it.nrows[t] - 1) / kPage + 1 : 0;
  }
  it.nmax = max(it.nkt[0], it.nkt[1]);
  return it;
}

__device__ __forceinline__ int pair_cost(const PrefillParams& p, int n, int ctx, int pair) {
  if (!lengths_ok(p, n, ctx)) return 0;
  int c = 0;
  for (int t = 0; t < 2; ++t) {
    const int q0 = pair * 256 + t * 128;
    const int nr = min(128, n - q0);
    if (nr > 0) c += (ctx - n + q0 + nr - 1) / kPage + 1;
  }
  return c;
}

// Greedy longest-first schedule: all items sorted by key-tile count
// (descending; ties in (sequence, pair, head) order), dealt to CTAs in a snake
// (0..N-1, N-1..0, ...).  Writes this CTA's items in order and returns their
// count, or -1 on every CTA when the launch is too large for the table
// (round-robin then).  Built by the 32 lanes of one warp, which all call it
// and get the same result: a pair at a time on one thread, the walk took most
// of the kernel's start-up.
//   scratch: 3 * kMaxCost ints (pairs per cost, first sorted position of each
//            cost, pairs of each cost placed so far)
//   seqs:    4 * B + 1 ints (chunk lengths, context lengths, first pair of
//            each sequence [B + 1], first packed token of each sequence)
__device__ int build_schedule(const PrefillParams& p, int* scratch, int* seqs, int* list, int N,
                              int c, int lane) {
  constexpr unsigned kAll = 0xffffffffu;
  const int maxc = 2 * p.max_pages + 1;
  if (maxc > kMaxCost || p.Hq > 256 || p.B > kMaxSchedSeqs) return -1;
  int* hist = scratch;
  int* start = scratch + kMaxCost;
  int* taken = scratch + 2 * kMaxCost;
  int* sn = seqs;
  int* sc = seqs + p.B;
  int* spf = seqs + 2 * p.B;
  int* stk = seqs + 3 * p.B + 1;
  for (int b = lane; b < maxc; b += 32) {
    hist[b] = 0;
    taken[b] = 0;
  }
  // lengths, then the pair and token prefix sums, 32 sequences at a time
  int64_t pbase = 0, tbase = 0;
  for (int s0 = 0; s0 < p.B; s0 += 32) {
    const int s = s0 + lane;
    int n = 0, ctx = 0;
    if (s < p.B) {
      n = __ldg(p.chunk_lens + s);
      ctx = __ldg(p.context_lens + s);
      sn[s] = n;
      sc[s] = ctx;
    }
    const int np = n > 0 ? n / 256 + (n % 256 != 0) : 0;  // < 2^24
    const int64_t tk = n > 0 ? n : 0;
    int inp = np;
    int64_t itk = tk;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(kAll, inp, o);
      const int64_t b = __shfl_up_sync(kAll, itk, o);
      if (lane >= o) {
        inp += a;
        itk += b;
      }
    }
    if (s < p.B) {
      spf[s] = (int)min(pbase + inp - np, (int64_t)INT32_MAX);
      stk[s] = (int)min(tbase + itk - tk, (int64_t)INT32_MAX);  // T < 2^31 for valid lengths
    }
    pbase += __shfl_sync(kAll, inp, 31);
    tbase += __shfl_sync(kAll, itk, 31);
  }
  // the table holds kMaxList items per CTA; the same test on every CTA
  const int64_t items = pbase * p.Hq;
  if (items > (int64_t)kMaxList * N) return -1;
  const int pairs = (int)pbase;  // from here on every count fits in 32 bits
  if (lane == 0) spf[p.B] = pairs;
  __syncwarp();
  // pair q's sequence: the last s with spf[s] <= q (sequences without pairs
  // have spf[s] == spf[s + 1])
  auto seq_of = [&](int q) {
    int lo = 0, hi = p.B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (spf[mid] <= q) lo = mid; else hi = mid;
    }
    return lo;
  };
  for (int q = lane; q < pairs; q += 32) {
    const int s = seq_of(q);
    atomicAdd(&hist[pair_cost(p, sn[s], sc[s], q - spf[s])], 1);
  }
  __syncwarp();
  // first sorted position of each cost: costs in decreasing order, Hq items
  // per pair (a scan over the buckets from the top, 32 at a time)
  int acc = 0;
  for (int b0 = maxc - 1; b0 >= 0; b0 -= 32) {
    const int b = b0 - lane;
    const int v = b >= 0 ? hist[b] * p.Hq : 0;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(kAll, inc, o);
      if (lane >= o) inc += a;
    }
    if (b >= 0) start[b] = acc + inc - v;
    acc += __shfl_sync(kAll, inc, 31);
  }
  __syncwarp();
  // each pair's rank among the pairs of its cost, in (sequence, pair) order,
  // 32 pairs at a time; its Hq items take the positions start + rank * Hq ...
  const int N2 = 2 * N;
  for (int q0 = 0; q0 < pairs; q0 += 32) {
    const int q = q0 + lane;
    const bool act = q < pairs;
    int s = 0, pr = 0, cost = -1;
    if (act) {
      s = seq_of(q);
      pr = q - spf[s];
      cost = pair_cost(p, sn[s], sc[s], pr);
    }
    const unsigned grp = __match_any_sync(kAll, cost);
    const int before = __popc(grp & ((1u << lane) - 1u));
    const int rank = act ? taken[cost] + before : 0;
    __syncwarp();
    if (act && before == 0) taken[cost] += __popc(grp);
    __syncwarp();
    if (!act) continue;
    const int pos0 = start[cost] + rank * p.Hq;
    for (int k = 0; k < 2; ++k) {
      // this CTA's positions of the snake: pos = res (mod 2N)
      const int res = k ? N2 - 1 - c : c;
      int d = (res - pos0) % N2;
      if (d < 0) d += N2;
      for (int pos = pos0 + d; pos < pos0 + p.Hq; pos += N2) {
        int* e = list + kListInts * (pos / N);
        e[0] = s;
        e[1] = (pr << 8) | (pos - pos0);
        e[2] = stk[s] + pr * 256;
        e[3] = sn[s];
        e[4] = sc[s];
      }
    }
  }
  __syncwarp();
  int rows = 0;  // snake rows that hold an item for this CTA (<= kMaxList)
  for (int r = 0; r <= kMaxList; ++r) {
    const int64_t pos = (int64_t)r * N + ((r & 1) ? N - 1 - c : c);
    if (pos >= items) break;
    ++rows;
  }
  return rows;
}

// Item source shared by all roles: the schedule table, or round-robin over
// (sequence, pair, head) when the table is unavailable.
struct ItemSource {
  const int* list;
  int count;  // -1: round-robin
  int s = 0, pairs_before = 0, tok_before = 0;
  __device__ bool get(const PrefillParams& p, int r, Item& it) {
    if (count >= 0) {
      if (r >= count) return false;
      const int* e = list + kListInts * r;
      it = make_item(p, e[0], e[1] >> 8, e[1] & 255, e[2], e[3], e[4]);
      return true;
    }
    const int i = (int)blockIdx.x + r * (int)gridDim.x;
    const int pair = i / p.Hq, g = i - pair * p.Hq;
    while (s < p.B) {
      const int n = __ldg(p.chunk_lens + s);
      const int np = n > 0 ? (n + 255) / 256 : 0;
      if (pair < pairs_before + np) break;
      pairs_before += np;
      tok_before += n > 0 ? n : 0;
      ++s;
    }
    if (s >= p.B) return false;
    const int pr = pair - pairs_before;
    it = make_item(p, s, pr, g, tok_before + pr * 256, __ldg(p.chunk_lens + s),
                   __ldg(p.context_lens + s));
    return true;
  }
};

// D[tmem] (+)= A[tmem] * B[smem]: A is M x 16 BF16 (lane = row, pairs per column).
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
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
  B.q_empty = bar + 2;
  B.k_full = bar + 4;
  B.k_empty = B.k_full + kRingK;
  B.v_full = B.k_empty + kRingK;
  B.v_empty = B.v_full + kRingV;
  B.s_full = B.v_empty + kRingV;
  B.p_full = B.s_full + 2;
  B.o_done = B.p_full + 2;
  B.o_free = B.o_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBars + kNumBars * 8);
  int* list_count = reinterpret_cast<int*>(tmem_slot + 1);
  int* list = reinterpret_cast<int*>(smem + kList);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&B.q_full[t], 1);
      mbar_init(&B.q_empty[t], 1);
    }
    for (int i = 0; i < kRingK; ++i) {
      mbar_init(&B.k_full[i], 1);
      mbar_init(&B.k_empty[i], 1);
    }
    for (int i = 0; i < kRingV; ++i) {
      mbar_init(&B.v_full[i], 1);
      mbar_init(&B.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B.s_full[i], 1);
      mbar_init(&B.p_full[i], 128);
      mbar_init(&B.o_done[i], 1);
      mbar_init(&B.o_free[i], 128);
    }
    fence_mbar_init();
  }
  if (warp == 0) {
    // the rings are idle until the first load: scratch for the schedule
    const int count = build_schedule(p, reinterpret_cast<int*>(smem + kK),
                                     reinterpret_cast<int*>(smem + kV), list, gridDim.x,
                                     blockIdx.x, lane);
    if (lane == 0) *list_count = count;
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  ItemSource src{list, *list_count};

  if (warp == 0 || warp == kVWarp) {
    // ------------------------------------------------------------ producers
    // warp 0: Q and K tiles; warp 10: V tiles.  Each runs ahead as far as its ring allows.
    if (lane == 0) {
      const bool is_k = warp == 0;
      const CUtensorMap* map = is_k ? &tm_k : &tm_v;
      const int ring_n = is_k ? kRingK : kRingV;
      uint64_t* full = is_k ? B.k_full : B.v_full;
      uint64_t* empty = is_k ? B.k_empty : B.v_empty;
      uint8_t* ring = smem + (is_k ? kK : kV);
      if (is_k) prefetch_tensor_map(&tm_q);
      prefetch_tensor_map(map);
      const uint64_t pol_kv = l2_policy_evict_last();  // reused by other tiles/heads
      const uint64_t pol_q = l2_policy_evict_first();
      uint32_t tiles = 0;
      uint32_t qitems[2] = {0, 0};  // items in which each query tile had key tiles
      bool ok = true;
      Item it;
      for (int r = 0; ok && src.get(p, r, it); ++r) {
        if (it.nmax == 0) continue;
        const int32_t* bt = p.block_table + (int64_t)it.s * p.max_pages;
        for (int kt = 0; kt < it.nmax; ++kt, ++tiles) {
          int page = __ldg(bt + kt);
          if (page < 0 || page >= p.num_pages) page = 0;  // sequence reported invalid
          const int slot = tiles % ring_n;
          const int x = it.h * kHeadDim, y = page * kPage;
          if (!(ok = mbar_wait(&empty[slot], ((tiles / ring_n) & 1) ^ 1, p.status))) break;
          mbar_arrive_expect_tx(&full[slot], kTileBytes);
          tma_load_2d(ring + slot * kTileBytes, map, x, y, &full[slot], pol_kv);
          tma_load_2d(ring + slot * kTileBytes + kBox, map, x + 64, y, &full[slot], pol_kv);
          if (is_k && kt == 0) {
            // each query tile's Q once its buffer is free (after the previous
            // item's last QK^T of that tile); the first K tile goes ahead of it
            for (int t = 0; t < 2 && ok; ++t) {
              if (it.nkt[t] == 0) continue;
              if (!(ok = mbar_wait(&B.q_empty[t], (qitems[t] & 1) ^ 1, p.status))) break;
              ++qitems[t];
              mbar_arrive_expect_tx(&B.q_full[t], kTileBytes);
              tma_load_3d(smem + kQ + t * kTileBytes, &tm_q, 0, it.g, it.tok0 + t * 128,
                          &B.q_full[t], pol_q);
              tma_load_3d(smem + kQ + t * kTileBytes + kBox, &tm_q, 64, it.g, it.tok0 + t * 128,
                          &B.q_full[t], pol_q);
            }
            if (!ok) break;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = umma_idesc_bf16(128, 128, false, false);
      const uint32_t idesc_pv = umma_idesc_bf16(128, 128, false, true);
      uint32_t tiles = 0;
      uint32_t gt[2] = {0, 0};     // key tiles each query tile has been through (all items)
      uint32_t gitems[2] = {0, 0};  // items in which each query tile had key tiles
      bool ok = true;
      auto qk = [&](int t, uint32_t kidx) {
        const uint32_t q_addr = smem_u32(smem + kQ + t * kTileBytes);
        const uint32_t k_addr = smem_u32(smem + kK + (kidx % kRingK) * kTileBytes);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t ad = umma_sdesc_sw128(q_addr + (k >> 2) * kBox + (k & 3) * 32, 16, 1024);
          const uint64_t bd = umma_sdesc_sw128(k_addr + (k >> 2) * kBox + (k & 3) * 32, 16, 1024);
          umma_bf16_ss(tmem + kColS + t * 128, ad, bd, idesc_qk, k > 0 ? 1u : 0u);
        }
        umma_commit(&B.s_full[t]);
      };
      auto pv = [&](int t, uint32_t kidx, bool first) -> bool {
        if (!mbar_wait(&B.p_full[t], gt[t] & 1, p.status)) return false;
        if (!mbar_wait(&B.v_full[kidx % kRingV], (kidx / kRingV) & 1, p.status)) return false;
        if (first && gitems[t] > 1 && !mbar_wait(&B.o_free[t], gitems[t] & 1, p.status))
          return false;
        tc_fence_after();
        const uint32_t v_addr = smem_u32(smem + kV + (kidx % kRingV) * kTileBytes);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t bd = umma_sdesc_sw128(v_addr + k * 2048, kBox, 1024);
          umma_bf16_ts(tmem + kColO + t * 128, tmem + kColS + t * 128 + k * 8, bd, idesc_pv,
                       (first && k == 0) ? 0u : 1u);
        }
        umma_commit(&B.o_done[t]);
        ++gt[t];
        return true;
      };
      auto wait_k = [&](uint32_t kidx) -> bool {
        const bool r = mbar_wait(&B.k_full[kidx % kRingK], (kidx / kRingK) & 1, p.status);
        tc_fence_after();
        return r;
      };
      Item it;
      for (int r = 0; ok && src.get(p, r, it); ++r) {
        if (it.nmax == 0) continue;
        const uint32_t k0 = tiles;
        if (!(ok = wait_k(k0))) break;
        for (int t = 0; t < 2 && ok; ++t) {
          if (it.nkt[t] == 0) continue;
          ++gitems[t];
          if (!(ok = mbar_wait(&B.q_full[t], (gitems[t] - 1) & 1, p.status))) break;
          tc_fence_after();
          qk(t, k0);
          if (it.nkt[t] == 1) umma_commit(&B.q_empty[t]);
        }
        if (!ok) break;
        umma_commit(&B.k_empty[k0 % kRingK]);
        for (int j = 0; j < it.nmax && ok; ++j) {
          const uint32_t kidx = k0 + j;
          const bool next = j + 1 < it.nmax;
          bool k_ready = false;
          if (j < it.nkt[0]) {
            if (!(ok = pv(0, kidx, j == 0))) break;
            if (j + 1 < it.nkt[0]) {
              if (!(ok = wait_k(kidx + 1))) break;
              k_ready = true;
              qk(0, kidx + 1);
              if (j + 2 == it.nkt[0]) umma_commit(&B.q_empty[0]);
            }
          }
          if (j < it.nkt[1]) {
            if (!(ok = pv(1, kidx, j == 0))) break;
          }
          umma_commit(&B.v_empty[kidx % kRingV]);
          if (j + 1 < it.nkt[1]) {
            if (!k_ready && !(ok = wait_k(kidx + 1))) break;
            qk(1, kidx + 1);
            if (j + 2 == it.nkt[1]) umma_commit(&B.q_empty[1]);
          }
          if (next) umma_commit(&B.k_empty[(kidx + 1) % kRingK]);
        }
        tiles += it.nmax;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax (query tile A or B)
    const int qtile = (warp - 2) >> 2;       // 0: warps 2-5 (tile A), 1: warps 6-9 (tile B)
    const int quarter = warp & 3;            // TMEM lanes this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int t = (warp - 2 - 4 * qtile) * 32 + lane;  // 0..127 within the group
    const uint32_t s_cols = tmem + lane_base + kColS + qtile * 128;
    const uint32_t o_cols = tmem + lane_base + kColO + qtile * 128;
    const float c = p.scale_log2;
    if (blockIdx.x == 0 && warp == 2 && p.status) {
      int sum = 0;
      for (int e = lane; e < p.B; e += 32) sum += max(__ldg(p.chunk_lens + e), 0);
#pragma unroll
      for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (lane == 0 && sum != p.T) atomicOr(p.status, PA_STATUS_BAD_TOKENS);
    }
    uint32_t tiles = 0, gt = 0;
    bool ok = true;
    Item it;
    for (int r = 0; ok && src.get(p, r, it); ++r) {
      const int nkt = it.nkt[qtile];
      const uint32_t k0 = tiles;
      if (it.nmax > 0) tiles += it.nmax;
      const bool reporter = qtile == 0 && t == 0 && it.pair == 0 && it.g == 0 && p.status;
      const int nrows = it.nrows[qtile];
      const int64_t tok = (int64_t)it.tok0 + qtile * 128 + row;
      const bool row_out = row < nrows && tok >= 0 && tok < p.T;
      uint8_t* dst = reinterpret_cast<uint8_t*>(p.out) +
                     ((tok * p.Hq + it.g) * kHeadDim) * (p.out_f32 ? 4 : 2);
      if (nkt == 0) {
        // tile A has key tiles unless the lengths are invalid
        if (!it.len_ok && reporter) atomicOr(p.status, PA_STATUS_BAD_LENGTH);
        if (row_out)  // lengths invalid: zero rows
          for (int cc = 0; cc < (p.out_f32 ? 32 : 16); ++cc)
            reinterpret_cast<uint4*>(dst)[cc] = make_uint4(0, 0, 0, 0);
        continue;
      }
      const int pos = it.prior + it.pair * 256 + qtile * 128 + min(row, nrows - 1);  // query position
      const int last_page = (it.ctx - 1) / kPage;
      const int vtail = it.ctx % kPage;  // rows >= vtail of the last page are past the context
      // the first P.V to read the last page zeroes its tail: tile A's if it reaches it
      const bool zero_mine = vtail != 0 && nkt - 1 == last_page &&
                             (qtile == 0 || it.nkt[0] - 1 != last_page);
      // block-table entries of the context: the first 32 loaded now, checked
      // after the key tiles (off the path to the first tile)
      const int used = (it.ctx + kPage - 1) / kPage;
      const int32_t* bt = p.block_table + (int64_t)it.s * p.max_pages;
      const int pg_first = lane < used ? __ldg(bt + lane) : 0;
      float m = -INFINITY, l = 0.f;
      for (int kt = 0; kt < nkt; ++kt, ++gt) {
        if (!(ok = mbar_wait_warp(&B.s_full[qtile], gt & 1, p.status))) break;
        tc_fence_after();
        // causal mask only where the tile crosses pos: masked scores take no part
        const int key0 = kt * kPage;
        const int nvis = min(max(pos - key0 + 1, 0), kPage);  // visible keys of this row
        // warp-uniform choices: the TMEM loads and stores below are .sync.aligned
        const bool diag = __any_sync(0xffffffffu, nvis < kPage);
        const float2 c2 = make_float2(c, c);
        if (__any_sync(0xffffffffu, m == -INFINITY)) {
          // the row's first key tile: the exact max of c * s over the visible keys
          float mx = -INFINITY;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t sr[32];
            tmem_ld32(s_cols + cc * 32, sr);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const float t = __uint_as_float(sr[e]) * c;
              mx = fmaxf(mx, cc * 32 + e < nvis ? t : -INFINITY);
            }
          }
          if (m == -INFINITY) m = mx;
        }
        // One pass, speculatively against the running reference m: p = 2^(c s - m),
        // tracking the largest exponent.  The reference moves (and the tile is
        // redone) only when some visible score exceeds it by more than 2^8.
        float alpha = 1.f;
        bool rescale = false;
        uint32_t pw[64];  // P as BF16 pairs
        float2 sum2;
        auto pass = [&](float m_ref, auto masked) -> float {
          const float2 nm2 = make_float2(-m_ref, -m_ref);
          float dmax = -INFINITY;
          sum2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t sr[32];
            tmem_ld32(s_cols + cc * 32, sr);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float2 d2 = __ffma2_rn(make_float2(__uint_as_float(sr[2 * e]),
                                                 __uint_as_float(sr[2 * e + 1])), c2, nm2);
              if (decltype(masked)::value) {
                const int k0e = cc * 32 + 2 * e;
                d2.x = k0e < nvis ? d2.x : -INFINITY;
                d2.y = k0e + 1 < nvis ? d2.y : -INFINITY;
              }
              dmax = fmaxf(dmax, fmaxf(d2.x, d2.y));
              const float2 p2 = make_float2(fast_exp2(d2.x), fast_exp2(d2.y));
              sum2 = __fadd2_rn(sum2, p2);
              pw[cc * 16 + e] = pack_bf16x2(p2.x, p2.y);
            }
          }
          return dmax;
        };
        const float m_use = m == -INFINITY ? 0.f : m;  // nothing visible yet: every p = 0
        const float dmax = diag ? pass(m_use, std::true_type{}) : pass(m_use, std::false_type{});
        const bool over = dmax > kRescaleThreshold;
        if (__any_sync(0xffffffffu, over)) {
          // rare: move this row's reference up to its tile max and redo the tile
          const float m_new = over ? m_use + dmax : m_use;
          if (over) {
            alpha = fast_exp2(-dmax);
            rescale = true;
            m = m_new;
          }
          if (diag) pass(m_new, std::true_type{}); else pass(m_new, std::false_type{});
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) w[e] = pw[cc * 16 + e];
          tmem_st16(s_cols + cc * 16, w);
        }
        l = l * alpha + (sum2.x + sum2.y);
        if (zero_mine && kt == nkt - 1) {
          // zero V rows past the context in the last page before P.V reads them
          const uint32_t kidx = k0 + kt;
          const int vs = kidx % kRingV;
          if (!(ok = mbar_wait_warp(&B.v_full[vs], (kidx / kRingV) & 1, p.status))) break;
          const int rr = vtail + t;
          if (rr < kPage) {
            const uint32_t vb = smem_u32(smem + kV + vs * kTileBytes) + rr * 128;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
              sts128(vb + ch * 16, 0u, 0u, 0u, 0u);
              sts128(vb + kBox + ch * 16, 0u, 0u, 0u, 0u);
            }
          }
          fence_proxy_async_smem();
        }
        // warp-uniform: lanes that need no rescale take alpha = 1 (exact)
        if (__any_sync(0xffffffffu, rescale) && kt > 0) {
          // O holds P.V up to the previous key tile: wait for it, then scale
          if (!(ok = mbar_wait_warp(&B.o_done[qtile], (gt - 1) & 1, p.status))) break;
          tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t orow[32];
            tmem_ld32(o_cols + cc * 32, orow);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) orow[e] = __float_as_uint(__uint_as_float(orow[e]) * alpha);
            tmem_st32(o_cols + cc * 32, orow);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&B.p_full[qtile]);
      }
      if (!ok) break;
      bool pg_bad = pg_first < 0 || pg_first >= p.num_pages;
      for (int e = lane + 32; e < used; e += 32) {
        const int pg = __ldg(bt + e);
        pg_bad |= (pg < 0 || pg >= p.num_pages);
      }
      const bool bad = __any_sync(0xffffffffu, pg_bad);
      if (bad && reporter) atomicOr(p.status, PA_STATUS_BAD_PAGE);
      // ---- epilogue: O / l for this row
      if (!(ok = mbar_wait_warp(&B.o_done[qtile], (gt - 1) & 1, p.status))) break;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      // an invalid sequence may have read a substitute page: select zeros
      const uint32_t keep = bad ? 0u : 0xffffffffu;
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t o0[32];
        tmem_ld32(o_cols + cc * 32, o0);
        tmem_wait_ld();
        if (row_out) {
          if (p.out_f32) {
            uint4* d4 = reinterpret_cast<uint4*>(dst) + cc * 8;
#pragma unroll
            for (int e = 0; e < 8; ++e)
              d4[e] = make_uint4(__float_as_uint(__uint_as_float(o0[4 * e]) * inv) & keep,
                                 __float_as_uint(__uint_as_float(o0[4 * e + 1]) * inv) & keep,
                                 __float_as_uint(__uint_as_float(o0[4 * e + 2]) * inv) & keep,
                                 __float_as_uint(__uint_as_float(o0[4 * e + 3]) * inv) & keep);
          } else {
            uint4* d4 = reinterpret_cast<uint4*>(dst) + cc * 4;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float* f = reinterpret_cast<const float*>(o0) + 8 * e;
              d4[e] = make_uint4(pack_bf16x2(f[0] * inv, f[1] * inv) & keep,
                                 pack_bf16x2(f[2] * inv, f[3] * inv) & keep,
                                 pack_bf16x2(f[4] * inv, f[5] * inv) & keep,
                                 pack_bf16x2(f[6] * inv, f[7] * inv) & keep);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&B.o_free[qtile]);
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
  static_assert(3 * kMaxCost * 4 <= kRingK * kTileBytes, "schedule scratch must fit the K ring");
  static_assert((4 * kMaxSchedSeqs + 1) * 4 <= kRingV * kTileBytes, "schedule lengths must fit the V ring");
  cudaError_t e =
      cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM (tensor memory and shared memory are sized for one)
  const int64_t max_items = ((int64_t)p.T / 256 + p.B) * p.Hq;
  const int grid = (int)(max_items < num_sms ? max_items : num_sms);
  if (grid < 1) return cudaSuccess;
  prefill_kernel<<<grid, kThreads, kSmem, stream>>>(tm_k, tm_v, tm_q, p);
  return cudaGetLastError();
}

}  // namespace pa
