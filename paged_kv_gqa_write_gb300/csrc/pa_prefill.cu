// pa_prefill.cu -- causal chunked-prefill attention over the paged cache on
// the 5th-generation tensor cores, one CTA pair (a cluster of two CTAs on two
// SMs) per work item, with pair MMAs (tcgen05 cta_group::2, M = 256).
//
// "Qwen3-14B" (pypto-lib), "prefill_fwd": per layer the KV cache update is
// followed by causal attention over token-major packed inputs
// (T = sum(chunk_lens)).  "Qwen 3" (TensorSharp), 4.1 "Attention": full
// causal GQA, no window or sinks.  New token j of sequence s sits at
// position ctx[s] - chunk_lens[s] + j and attends to keys 0..position of its
// own sequence, read from the paged cache (prior context plus the chunk,
// which pa_kv_write has already stored).
//
// Work item: (sequence, pair of consecutive 128-token query tiles, query
// head).  CTA r of the pair owns query tile r: its 128 rows of Q, S, P and O.
// Per key page tile (one "step") the even CTA issues two pair products:
//   S = Q K^T   M = 256 (both tiles), N = 128 keys, K = 128 dims
//   O += P V    M = 256, N = 128 dims, K = 128 keys
// Each CTA stages only half of the page tile: keys 64r..64r+63 of K (the
// half of S's N columns the pair product takes from it) and dims 64r..64r+63
// of V (the half of O's N columns), so one 64 KB page tile feeds four
// 128x128x128 products while each SM reads 32 KB of it.
//  * warp 0 (one lane): Q tiles (double-buffered: the next item's tile loads
//    during this one) and K halves (3-stage ring: stage j % 3 is free once
//    S(j - 3) is done).  Both CTAs' loads complete on the even CTA's
//    barriers (paired TMA), which its S issuer waits on.
//  * warp 10 (one lane): V halves (3-stage ring, free once P.V(j - 3) is
//    done), completing locally.
//  * warp 1: both CTAs allocate tensor memory together (S0, S1, S2, O).  In
//    the even CTA one lane of warp 1 and one of warp 11 issue the MMAs,
//    taking alternate steps: each issues P.V(j) and then S(j + 3), so each
//    one's waits and commits overlap the other's products in the tensor
//    core's queue.  S is triple-buffered, so the scores of the next steps are
//    computed while the softmax works, and P(j) is written back over S(j) (A
//    operand from tensor memory), so the softmax runs up to three steps ahead
//    of P.V; one thread's products execute in issue order, so S(j + 3)
//    follows P.V(j) without waiting for it.
//  * warps 2-9: softmax and epilogue, two threads per query row (warps w and
//    w + 4 share the row's tensor-memory lanes; each takes 64 of the 128
//    columns).  Per step: tcgen05.ld of the score half-row, causal mask (only
//    on tiles that cross the row's position), online softmax in the log2
//    domain against a running reference that moves only when a score exceeds
//    it by 2^8 (the two halves agree on it through shared memory; O is then
//    rescaled in tensor memory), P rounded to BF16 pairs into the first 32
//    of the half's own 64 S columns, and the row sum taken over the rounded
//    weights the MMA uses.  The warps then wait for this CTA's V half, zero
//    its rows past the context on the sequence's last page (P is 0 there,
//    but 0 * NaN is NaN), and arrive on the even CTA's P barrier: the P.V
//    product reads both CTAs' P and V halves.
// Waits on barriers completed by tensor-core commits (multicast to both CTAs)
// or by copies take acquire at CTA scope, as for a single CTA; the waits on
// the even CTA's P barrier, which the odd CTA's threads arrive on, take it at
// cluster scope.  (A cluster-scope acquire cost 0.1-0.2 us per wait.)
// "P ready" crosses the pair once per step.  Each odd-CTA warp completes its
// tensor-memory stores (tcgen05.wait::st, then tcgen05.fence before the
// thread synchronisation), makes its shared-memory writes visible to the
// tensor core (fence.proxy.async), and arrives on the even CTA's barrier
// after a cluster-scope release restricted to shared memory: a full
// cluster-scope release waits for global memory and cost about 0.6 us per
// arrival, the restricted one about as much as a local arrival.
// FP8 cache (e4m3 codes, per-KV-head scales): the K halves land as e4m3 by
// the same paired TMA and S = Q K^T runs on them (kind::f8f6f4); four
// converter warps split each query row, times a power of two of its own, into
// e4m3 hi and lo rows in the place of the BF16 tile's two boxes (S = hi K^T +
// lo K^T, 8 products per step as with BF16), and rewrite the V halves as F16
// for P.V (kind::f16, P in F16).
// Epilogue: O / l per row.  A full 128-row tile with BF16 output is staged in
// shared memory (128-byte swizzle) and written by one TMA tensor store that
// runs on while the warps start the next item; partial tiles and FP32 output
// are written row by row.
// Key pages entirely above both tiles' last query positions are never loaded
// (causal tile skipping); the lower tile sees its pair's last page fully
// masked.  Items are dealt to the pairs in decreasing order of key-tile
// count, snaking across pairs (a greedy longest-first balance every CTA
// computes from the lengths); very large launches fall back to round-robin.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <type_traits>

#include "pa_launch.cuh"

namespace pa {
namespace {

constexpr int kSoftWarp0 = 2;                 // softmax warps 2 .. 9
constexpr int kSoftmaxWarps = 8;
constexpr int kVWarp = 10;                    // V producer
constexpr int kPvWarp = 11;                   // P.V issuer (even CTA)
constexpr int kConvWarp0 = 12;                // FP8 cache: converter warps 12 .. 15
constexpr int kQBytes = 128 * 128 * 2;        // one query tile (two 64-column boxes)
constexpr int kQBox = 16384;
constexpr int kKBytes = 64 * 128 * 2;         // this CTA's K half: 64 keys x 128 dims
constexpr int kKBox = 8192;                   // 64 keys x 64 dims
constexpr int kVBytes = 128 * 64 * 2;         // this CTA's V half: 128 keys x 64 dims
constexpr int kK8Bytes = 64 * 128;            // the same K half as e4m3 codes
constexpr int kV8Bytes = 128 * 64;            // the same V half as e4m3 codes
constexpr int kNumS = 3;                      // S buffers in tensor memory
constexpr int kMaxList = PA_PREFILL_SCHEDULE_ITEMS;  // scheduled items per pair
constexpr int kOutBytes = 128 * 128 * 2;
constexpr int kOutBox = 16384;
constexpr int kListInts = 5;                  // per item: s, pair|head, tok0, chunk len, ctx
constexpr int kMaxCost = 4096;                // schedule histogram buckets
constexpr int kSchedBytes = 3 * kMaxCost * 4; // the schedule's scratch ...
constexpr int kSeqBytes = 48 * 1024;          // ... and its staged lengths
constexpr int kMaxSchedSeqs = (kSeqBytes / 4 - 1) / 4;  // sequences the schedule stages
// Shared memory layout (offsets from a 1024-aligned base; identical in both
// CTAs: a pair MMA reads both at the same offsets).  3-stage K ring (BF16, or
// the e4m3 codes themselves with the FP8 cache), S(j) done frees K stage
// j % 3.  BF16 cache: 3-stage V operand ring, P.V(j) done frees V stage j % 3.
// FP8 cache: the V operand ring holds F16, filled by the converter warps
// from a 3-stage ring of e4m3 V halves; the query tile holds the e4m3 hi and lo
// halves of the split (below) in the place of the BF16 tile's two boxes.
template <bool FP8>
struct Lay {
  static constexpr int kThreads = (FP8 ? kConvWarp0 + 4 : kPvWarp + 1) * 32;
  static constexpr int kRingK = 3, kRingV = 3;  // operand stages
  static constexpr int kKStage = FP8 ? kK8Bytes : kKBytes;
  static constexpr int kRing8 = FP8 ? 3 : 0;               // e4m3 V stages
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + 2 * kQBytes;
  static constexpr int kV = kK + kRingK * kKStage;
  static constexpr int kV8 = kV + kRingV * kVBytes;
  static constexpr int kOut = kV8 + kRing8 * kV8Bytes;  // BF16 output tile staging: 2 boxes of 128 x 64
  static constexpr int kX = kOut + kOutBytes;           // row exchange between the two halves: [2][128] float
  // FP8: 1 / x per query row, [4][128] float by item ordinal mod 4 (a slot
  // is rewritten four items later, when the softmax is past the item after it)
  static constexpr int kQInv = kX + 2 * 128 * 4;
  static constexpr int kList = kQInv + (FP8 ? 4 * 128 * 4 : 0);  // schedule [kMaxList][kListInts] int
  static constexpr int kBars = kList + kMaxList * kListInts * 4;
  // q_full, q_empty, k_full, v_full, s_full, p_full, o_done, drain; FP8:
  // q16_full, qs_full, v16_full, v8_full, v8_empty
  static constexpr int kNumBars = 2 + 2 + kRingK + kRingV + 3 * kNumS + 1 +
                                  (FP8 ? 2 + 4 + kRingV + 2 * kRing8 : 0);
  static constexpr int kSmem = kBars + kNumBars * 8 + 16 + 1024;
  // the buffers are idle until the first load: scratch for the schedule
  static constexpr int kSched = FP8 ? kQ : kK;
  static constexpr int kSeqs = FP8 ? kQ + kSchedBytes : kV;
  static_assert(kSched + kSchedBytes <= kSeqs, "schedule scratch must fit the operand rings");
  static_assert(kSeqs + kSeqBytes <= kOut, "schedule lengths must fit the rings");
  static_assert(kSmem <= 232448, "prefill shared memory exceeds the per-CTA limit");
};
// TMEM columns (the same in both CTAs)
constexpr uint32_t kColS = 0;     // S0, S1, S2: 128 columns each, by step mod 3; P(j) over S(j)
constexpr uint32_t kColO = 384;   // O: 128 columns
// P(j) as BF16 pairs inside S(j): keys 0-63 (half 0) in columns 0-31, keys
// 64-127 (half 1) in columns 64-95, each half writing over its own scores
__host__ __device__ constexpr uint32_t p_col(int kstep) {
  return kstep < 4 ? kstep * 8 : 64 + (kstep - 4) * 8;
}
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;     // log2 units
constexpr uint16_t kPairMask = 3;             // both CTAs of the cluster
constexpr uint64_t kDrainLimitNs = 100000000ull;  // copies land in microseconds

// Instruction descriptor of tcgen05.mma kind::f8f6f4 with E4M3 A and B (format
// code 0), both K-major, FP32 accumulate, an M x N tile.
__host__ __device__ constexpr uint32_t umma_idesc_e4m3(int M, int N) {
  return (1u << 4)                            // D format: F32
         | ((uint32_t)(N >> 3) << 17)         // N / 8
         | ((uint32_t)(M >> 4) << 24);        // M / 16
}

// D (+)= A * B over 32 e4m3 elements of K across a CTA pair (cta_group::2,
// M = 256), operands in both CTAs' shared memory as umma_bf16_ss_pair takes them.
__device__ __forceinline__ void umma_e4m3_ss_pair(uint32_t d_tmem, uint64_t a_desc,
                                                  uint64_t b_desc, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct Bars {
  uint64_t* q_full;   // [2] even CTA: both CTAs' query tiles landed
  uint64_t* q_empty;  // [2] the item's last S product read the tile
  uint64_t* k_full;   // [3] even CTA: both K halves landed
  uint64_t* v_full;   // [3] this CTA's V half landed
  uint64_t* s_full;   // [3] S(g) in buffer g % 3 done (and K stage g % 3 free)
  uint64_t* p_full;   // [3] even CTA: P(g) written in both CTAs, V(g) halves in place
  uint64_t* o_done;   // [3] P.V(g) done: O holds every step <= g, V stage g % 3 free
  uint64_t* drain;    // every MMA issued (by both issuers) has completed
  // FP8 cache (q_full then completes per CTA: each loads its own tile)
  uint64_t* q16_full;  // [2] even CTA: both CTAs' query tiles split into e4m3 hi / lo
  uint64_t* qs_full;   // [4] this CTA's 1 / x per query row stored (item ordinal mod 4)
  uint64_t* v16_full;  // [2] this CTA's V half converted to F16
  uint64_t* v8_full;   // [3] this CTA's e4m3 V half landed
  uint64_t* v8_empty;  // [3] ... converted
};

struct Item {
  int s, g, h, pair;
  int tok0;          // packed index of the pair's first query token
  int nrows[2];      // query rows of tiles 0, 1 (<= 128; tile 1 may be 0)
  int nkt[2];        // key tiles each query tile sees (0: none / lengths invalid)
  int nmax;          // key tiles (steps) the pair runs
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

// Key tiles a pair runs: its two query tiles go through the key tiles in
// lockstep (one M = 256 product per step), so the longer tile's count.
__device__ __forceinline__ int pair_cost(const PrefillParams& p, int n, int ctx, int pair) {
  if (!lengths_ok(p, n, ctx)) return 0;
  int c = 0;
  for (int t = 0; t < 2; ++t) {
    const int q0 = pair * 256 + t * 128;
    const int nr = min(128, n - q0);
    if (nr > 0) c = max(c, (ctx - n + q0 + nr - 1) / kPage + 1);
  }
  return c;
}

// Greedy longest-first schedule: all items sorted by key-tile count
// (descending; ties in (sequence, pair, head) order), dealt to the N CTA pairs
// in a snake (0..N-1, N-1..0, ...).  Writes pair c's items in order and
// returns their count, or -1 on every CTA when the launch is too large for
// the table (round-robin then).  Both CTAs of a pair build the same list.  Built by the 32 lanes of one warp, which all call it
// and get the same result: a pair at a time on one thread, the walk took most
// of the kernel's start-up.
//   scratch: 3 * kMaxCost ints (pairs per cost, first sorted position of each
//            cost, pairs of each cost placed so far)
//   seqs:    4 * B + 1 ints (chunk lengths, context lengths, first pair of
//            each sequence [B + 1], first packed token of each sequence)
__device__ int build_schedule(const PrefillParams& p, int* scratch, int* seqs, int* list, int N,
                              int c, int lane) {
  constexpr unsigned kAll = 0xffffffffu;
  const int maxc = p.max_pages + 2;
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
// (sequence, pair, head) across the N pairs when the table is unavailable.
// A source walks its items in increasing r.
struct ItemSource {
  const int* list;
  int count;  // -1: round-robin
  int c, N;   // this pair, pairs in the launch
  int s = 0, pairs_before = 0, tok_before = 0;
  __device__ bool get(const PrefillParams& p, int r, Item& it) {
    if (count >= 0) {
      if (r >= count) return false;
      const int* e = list + kListInts * r;
      it = make_item(p, e[0], e[1] >> 8, e[1] & 255, e[2], e[3], e[4]);
      return true;
    }
    const int64_t i64 = (int64_t)c + (int64_t)r * N;
    if (i64 > INT32_MAX) return false;
    const int i = (int)i64;
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
  // Next item with key tiles (r advanced past it); false at the end.
  __device__ bool next_with_tiles(const PrefillParams& p, int& r, Item& it) {
    while (get(p, r, it)) {
      ++r;
      if (it.nmax > 0) return true;
    }
    return false;
  }
};

// Waits for the last phase of each barrier that saw `issued` loads spread
// round-robin over `n` barriers (no wait for barriers that saw none): every
// copy in flight lands before the shared memory is released.
__device__ __forceinline__ void drain_loads(uint64_t* bars, int n, uint32_t issued, int32_t* status,
                                            bool cluster_scope) {
  for (int i = 0; i < n; ++i) {
    const uint32_t cnt = issued > (uint32_t)i ? (issued - 1 - i) / n + 1 : 0;
    if (cnt == 0) continue;
    if (cluster_scope) mbar_wait_cl_for(&bars[i], (cnt - 1) & 1, status, kDrainLimitNs);
    else mbar_wait_for(&bars[i], (cnt - 1) & 1, status, kDrainLimitNs);
  }
}

template <bool FP8>
__global__ void __launch_bounds__(Lay<FP8>::kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o,
                   const PrefillParams p) {
  using L = Lay<FP8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kBars);
  Bars B;
  B.q_full = bar;
  B.q_empty = bar + 2;
  B.k_full = bar + 4;
  B.v_full = B.k_full + L::kRingK;
  B.s_full = B.v_full + L::kRingV;
  B.p_full = B.s_full + kNumS;
  B.o_done = B.p_full + kNumS;
  B.drain = B.o_done + kNumS;
  if constexpr (FP8) {
    B.q16_full = B.drain + 1;
    B.qs_full = B.q16_full + 2;
    B.v16_full = B.qs_full + 4;
    B.v8_full = B.v16_full + L::kRingV;
    B.v8_empty = B.v8_full + L::kRing8;
  }
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBars + L::kNumBars * 8);
  int* list_count = reinterpret_cast<int*>(tmem_slot + 1);
  int* list = reinterpret_cast<int*>(smem + L::kList);
  float* xch = reinterpret_cast<float*>(smem + L::kX);
  float* qinv = reinterpret_cast<float*>(smem + L::kQInv);  // FP8 only

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // query tile of the pair this CTA owns
  const bool even = rank == 0;              // issues the pair MMAs
  const int npairs = (int)cluster_count_x(), pair_id = (int)cluster_id_x();
  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&B.q_full[t], 1);
      mbar_init(&B.q_empty[t], 2);  // one commit from each MMA issuer
    }
    for (int i = 0; i < L::kRingK; ++i) mbar_init(&B.k_full[i], 1);
    for (int i = 0; i < L::kRingV; ++i) mbar_init(&B.v_full[i], 1);
    for (int i = 0; i < kNumS; ++i) {
      mbar_init(&B.s_full[i], 1);
      mbar_init(&B.p_full[i], 2 * kSoftmaxWarps);  // the softmax warps of both CTAs
      mbar_init(&B.o_done[i], 1);
    }
    mbar_init(B.drain, 2);  // one commit from each issuer
    if constexpr (FP8) {
      for (int i = 0; i < 2; ++i) mbar_init(&B.q16_full[i], 8);  // 4 converter warps x 2 CTAs
      for (int i = 0; i < 4; ++i) mbar_init(&B.qs_full[i], 4);
      for (int i = 0; i < L::kRingV; ++i) mbar_init(&B.v16_full[i], 4);
      for (int i = 0; i < L::kRing8; ++i) {
        mbar_init(&B.v8_full[i], 1);
        mbar_init(&B.v8_empty[i], 4);
      }
    }
    fence_mbar_init();
  }
  // Launched as a programmatic dependent of the kernel before it on the
  // stream (the chunk's KV write): the barrier set-up above touches only this
  // CTA's shared memory; everything from here on comes after that kernel has
  // completed and its writes are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (warp == 0) {
    // the rings are idle until the first load: scratch for the schedule
    const int count = build_schedule(p, reinterpret_cast<int*>(smem + L::kSched),
                                     reinterpret_cast<int*>(smem + L::kSeqs), list, npairs, pair_id,
                                     lane);
    if (lane == 0) *list_count = count;
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  // both CTAs' barriers are initialised before any paired copy, multicast
  // commit or remote arrival targets them
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  ItemSource src{list, *list_count, pair_id, npairs};

  if (warp == 0 || warp == kVWarp) {
    // ------------------------------------------------------------ producers
    if (lane == 0) {
      const bool is_k = warp == 0;
      if (is_k) prefetch_tensor_map(&tm_q);
      prefetch_tensor_map(is_k ? &tm_k : &tm_v);
      const uint64_t pol_kv = l2_policy_evict_last();  // reused by the other heads' items
      const uint64_t pol_q = l2_policy_evict_first();
      uint32_t tiles = 0, qitems = 0;
      bool ok = true;
      Item it;
      int r = 0;
      while (ok && src.next_with_tiles(p, r, it)) {
        const int32_t* bt = p.block_table + (int64_t)it.s * p.max_pages;
        if (is_k) {
          // this CTA's query tile, once the item two back released the buffer
          const int qb = qitems & 1;
          if (!(ok = mbar_wait(&B.q_empty[qb], ((qitems >> 1) & 1) ^ 1, p.status))) break;
          ++qitems;
          const int z = it.tok0 + (int)rank * 128;
          uint8_t* qdst = smem + L::kQ + qb * kQBytes;
          if constexpr (FP8) {
            // each CTA's own barrier: its converter warps rewrite the tile as F16
            mbar_arrive_expect_tx(&B.q_full[qb], kQBytes);
            tma_load_3d(qdst, &tm_q, 0, it.g, z, &B.q_full[qb], pol_q);
            tma_load_3d(qdst + kQBox, &tm_q, 64, it.g, z, &B.q_full[qb], pol_q);
          } else {
            if (even) mbar_arrive_expect_tx(&B.q_full[qb], 2 * kQBytes);
            const uint32_t qbar = mapa_shared(smem_u32(&B.q_full[qb]), 0);
            tma_load_3d_pair(qdst, &tm_q, 0, it.g, z, qbar, pol_q);
            tma_load_3d_pair(qdst + kQBox, &tm_q, 64, it.g, z, qbar, pol_q);
          }
        }
        for (int kt = 0; kt < it.nmax; ++kt, ++tiles) {
          int page = __ldg(bt + kt);
          if (page < 0 || page >= p.num_pages) page = 0;  // sequence reported invalid
          const int y = page * kPage;
          if (is_k) {
            // keys 64 rank .. + 63 of the page; stage tiles % 3 is free once
            // S(tiles - 3) is done.  FP8: the e4m3 half (128 one-byte dims, one
            // 128-byte-swizzled box) is QK^T's operand as it lands
            const int st = tiles % L::kRingK;
            if (tiles >= (uint32_t)L::kRingK &&
                !(ok = mbar_wait(&B.s_full[st], ((tiles / L::kRingK) & 1) ^ 1, p.status)))
              break;
            if (even) mbar_arrive_expect_tx(&B.k_full[st], 2 * L::kKStage);
            const uint32_t kbar = mapa_shared(smem_u32(&B.k_full[st]), 0);
            uint8_t* dst = smem + L::kK + st * L::kKStage;
            tma_load_2d_pair(dst, &tm_k, it.h * kHeadDim, y + (int)rank * 64, kbar, pol_kv);
            if constexpr (!FP8)
              tma_load_2d_pair(dst + kKBox, &tm_k, it.h * kHeadDim + 64, y + (int)rank * 64, kbar,
                               pol_kv);
          } else if constexpr (FP8) {
            // e4m3 V half: dims 64 rank .. + 63 of the 128 keys; stage tiles % 3
            // is free once the converter warps have read it
            const int st = tiles % L::kRing8;
            const uint32_t ph = ((tiles / L::kRing8) & 1) ^ 1;
            if (tiles >= (uint32_t)L::kRing8 && !(ok = mbar_wait(&B.v8_empty[st], ph, p.status)))
              break;
            mbar_arrive_expect_tx(&B.v8_full[st], kV8Bytes);
            tma_load_2d(smem + L::kV8 + st * kV8Bytes, &tm_v, it.h * kHeadDim + (int)rank * 64, y,
                        &B.v8_full[st], pol_kv);
          } else {
            // stage tiles % 3 is free once P.V(tiles - 3) is done
            const int st = tiles % L::kRingV;
            if (tiles >= (uint32_t)L::kRingV &&
                !(ok = mbar_wait(&B.o_done[st], ((tiles / L::kRingV) & 1) ^ 1, p.status)))
              break;
            mbar_arrive_expect_tx(&B.v_full[st], kVBytes);
            tma_load_2d(smem + L::kV + st * kVBytes, &tm_v, it.h * kHeadDim + (int)rank * 64, y,
                        &B.v_full[st], pol_kv);
          }
        }
      }
      // copies still in flight (only after a timeout) land before teardown;
      // the even CTA's barriers count both CTAs' Q and K halves
      if (!is_k) {
        if constexpr (FP8) drain_loads(B.v8_full, L::kRing8, tiles, p.status, false);
        else drain_loads(B.v_full, L::kRingV, tiles, p.status, false);
      } else {
        if (FP8) drain_loads(B.q_full, 2, qitems, p.status, false);  // each CTA's own
        else if (even) drain_loads(B.q_full, 2, qitems, p.status, true);
        if (even) drain_loads(B.k_full, L::kRingK, tiles, p.status, true);
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == kPvWarp) {
    if (even && lane == 0) {
      // ---------------------------------------------------------- MMA issuers (even CTA)
      // Two threads take alternate steps g (thread par takes g % 2 == par):
      // each issues P.V(g) and then S(g + 3), into the buffer that holds P(g).
      // One thread's products execute in issue order, so S(g + 3) runs after
      // P.V(g) has read P(g) without waiting for it, and the tensor core's
      // queue holds P.V(g), S(g + 3), P.V(g + 1), S(g + 4), ...  P.V(g) first
      // waits for P.V(g - 1) (the other thread's) to complete, which orders
      // the accumulation into O.  Thread 0 issues S(0..2) up front.
      const uint32_t par = warp == 1 ? 0u : 1u;
      // Q, K: K-major (FP8: e4m3 x e4m3, kind::f8f6f4); P (TMEM), V MN-major
      // (FP8: F16)
      const uint32_t idesc_qk = FP8 ? umma_idesc_e4m3(256, 128)
                                    : umma_idesc_bf16(256, 128, false, false);
      const uint32_t idesc_pv = FP8 ? umma_idesc_f16(256, 128, false, true)
                                    : umma_idesc_bf16(256, 128, false, true);
      bool ok = true;
      // S cursor: step gq of item iq (key tile jq), its query tile's ordinal qi
      ItemSource sq = src;
      int rq = 0, jq = 0;
      Item iq;
      bool hq = sq.next_with_tiles(p, rq, iq);
      uint32_t gq = 0, qi = 0, q_waited = ~0u;
      auto next_qk = [&](bool issue) {
        const int qb = qi & 1;
        if (issue) {
          if (q_waited != qi) {
            // FP8: both CTAs' tiles split into e4m3 hi and lo by their converter warps
            if (!(ok = FP8 ? mbar_wait_cl(&B.q16_full[qb], (qi >> 1) & 1, p.status)
                           : mbar_wait(&B.q_full[qb], (qi >> 1) & 1, p.status)))
              return;
            q_waited = qi;
          }
          const int sb = gq % kNumS, kb = gq % L::kRingK;
          const uint32_t kph = (gq / L::kRingK) & 1;
          if (!(ok = mbar_wait(&B.k_full[kb], kph, p.status))) return;
          tc_fence_after();
          const uint32_t qa = smem_u32(smem + L::kQ + qb * kQBytes);
          const uint32_t ka = smem_u32(smem + L::kK + kb * L::kKStage);
          const uint32_t d = tmem + kColS + sb * 128;
          if constexpr (FP8) {
            // S = (hi + lo) K^T: the hi rows (box 0) then the lo rows (box 1)
            // against the same e4m3 K half, 32 dims per instruction
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint64_t ad = umma_sdesc_sw128(qa + (k >> 2) * kQBox + (k & 3) * 32, 16, 1024);
              const uint64_t bd = umma_sdesc_sw128(ka + (k & 3) * 32, 16, 1024);
              umma_e4m3_ss_pair(d, ad, bd, idesc_qk, k > 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint64_t ad = umma_sdesc_sw128(qa + (k >> 2) * kQBox + (k & 3) * 32, 16, 1024);
              const uint64_t bd = umma_sdesc_sw128(ka + (k >> 2) * kKBox + (k & 3) * 32, 16, 1024);
              umma_bf16_ss_pair(d, ad, bd, idesc_qk, k > 0 ? 1u : 0u);
            }
          }
          umma_commit_pair(&B.s_full[sb], kPairMask);
        }
        ++gq;
        if (++jq == iq.nmax) {
          // the query tile is free once both threads' S products of the item
          // are done: each thread commits when its cursor leaves the item
          umma_commit_pair(&B.q_empty[qb], kPairMask);
          ++qi;
          jq = 0;
          hq = sq.next_with_tiles(p, rq, iq);
        }
      };
      for (int i = 0; i < kNumS && hq && ok; ++i) next_qk(par == 0);
      // P.V cursor
      ItemSource sp = src;
      int rp = 0;
      Item ip;
      uint32_t g = 0;
      while (ok && sp.next_with_tiles(p, rp, ip)) {
        for (int kt = 0; kt < ip.nmax && ok; ++kt, ++g) {
          const bool mine = (g & 1u) == par;
          if (mine) {
            // both CTAs' P (tensor memory) and V halves are in place, and
            // P.V(g - 1) has accumulated into O
            const int sb = g % kNumS;
            if (!(ok = mbar_wait_cl(&B.p_full[sb], (g / kNumS) & 1, p.status))) break;
            if (g > 0) {
              const uint32_t g1 = g - 1;
              if (!(ok = mbar_wait(&B.o_done[g1 % kNumS], (g1 / kNumS) & 1, p.status))) break;
            }
            tc_fence_after();
            const uint32_t va = smem_u32(smem + L::kV + (g % L::kRingV) * kVBytes);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint64_t bd = umma_sdesc_sw128(va + k * 2048, kVBytes, 1024);
              umma_bf16_ts_pair(tmem + kColO, tmem + kColS + sb * 128 + p_col(k), bd, idesc_pv,
                                (kt > 0 || k > 0) ? 1u : 0u);
            }
            umma_commit_pair(&B.o_done[sb], kPairMask);
          }
          // S(g + 3): by the thread that issued P.V(g)
          if (hq) next_qk(mine);
        }
      }
      // every product issued completes before the columns are released
      umma_commit_pair(B.drain, kPairMask);
    }
    __syncwarp();
    if (warp == 1 && lane == 0) mbar_wait_cl_for(B.drain, 0, p.status, kWaitLimitNs);
    __syncwarp();
  } else if (warp >= kConvWarp0) {
    // ------------------------------------------------------------ FP8 converters
    // Four warps (128 threads) per CTA.  Per item: this CTA's query tile, row
    // ct, times a power of two x_ct that brings the row's largest |q| into
    // [128, 256), split into two e4m3 rows hi = e4m3(x q) (box 0 of the tile)
    // and lo = e4m3(x q - hi) (box 1), in place; hi + lo = x q exactly for
    // every element of magnitude at least 2^-10 of the row's largest (a bf16
    // value has 8 significant bits, and the residual of its rounding to 4 is a
    // multiple of its last bit with at most 4 significant bits), smaller ones
    // are off by at most 2^-10 / x.  1 / x goes to the softmax.  QK^T then
    // runs on the e4m3 K halves as TMA lands them.  Per step: this CTA's e4m3
    // V half (thread = key) to F16 in the swizzled layout the BF16 path gets
    // from TMA (e4m3 values are exact in F16); a V stage is reused three
    // steps later, once P.V(j - 3) is done.  The even CTA's issuer waits for both
    // CTAs' query splits (remote arrivals from the odd CTA); V is this CTA's,
    // behind the softmax's P barrier.
    if constexpr (FP8) {
      const int ct = threadIdx.x - kConvWarp0 * 32;  // 0..127
      uint32_t q16_even[2];
      for (int i = 0; i < 2; ++i) q16_even[i] = mapa_shared(smem_u32(&B.q16_full[i]), 0);
      uint32_t tiles = 0, qitems = 0;
      bool ok = true;
      Item it;
      int r = 0;
      while (src.next_with_tiles(p, r, it)) {
        // ---- Q: row ct of this CTA's tile (16 chunks of 8 BF16 values, two
        // boxes) into e4m3 hi (box 0) and lo (box 1), in place
        const int qb = qitems & 1;
        if (ok) ok = mbar_wait_warp(&B.q_full[qb], (qitems >> 1) & 1, p.status);
        ++qitems;
        {
          const uint32_t qrow = smem_u32(smem + L::kQ + qb * kQBytes) + ct * 128;
          uint32_t w[64];  // the row's 128 BF16 values
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const uint4 v = lds128(qrow + (c >> 3) * kQBox + ((((uint32_t)c & 7) ^ (ct & 7)) << 4));
            w[4 * c] = v.x;
            w[4 * c + 1] = v.y;
            w[4 * c + 2] = v.z;
            w[4 * c + 3] = v.w;
          }
          // the largest magnitude (BF16 bits: the magnitude order is the
          // integer order; from 0x7f80 up: inf or NaN)
          uint32_t amax = 0;
#pragma unroll
          for (int e = 0; e < 64; ++e) amax = max(amax, max(w[e] & 0x7fffu, (w[e] >> 16) & 0x7fffu));
          float x, xinv = 1.f;
          if (amax >= 0x7f80u) {
            // inf or NaN in q: flagged, and the row's scores become NaN
            x = __uint_as_float(0x7fc00000u);
            if (p.status) atomicOr(p.status, PA_STATUS_Q_RANGE);
          } else {
            // largest = 1.f x 2^(be - 127); x = 2^(134 - be), kept a normal float
            const int sx = min(134 - (int)(amax >> 7), 126);
            x = __uint_as_float((uint32_t)(127 + sx) << 23);
            xinv = __uint_as_float((uint32_t)(127 - sx) << 23);
          }
#pragma unroll
          for (int c = 0; c < 8; ++c) {  // dims 16 c .. 16 c + 15
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              uint32_t h4 = 0, l4 = 0;
#pragma unroll
              for (int f = 0; f < 2; ++f) {
                const float2 a = bf16x2_to_float2(w[8 * c + 2 * e + f]);
                const float2 ax = make_float2(a.x * x, a.y * x);
                const __nv_fp8x2_storage_t h = __nv_cvt_float2_to_fp8x2(ax, __NV_SATFINITE, __NV_E4M3);
                const __half2 hh(__nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3));
                const float2 hf = __half22float2(hh);
                const __nv_fp8x2_storage_t l = __nv_cvt_float2_to_fp8x2(
                    make_float2(ax.x - hf.x, ax.y - hf.y), __NV_SATFINITE, __NV_E4M3);
                h4 |= (uint32_t)h << (16 * f);
                l4 |= (uint32_t)l << (16 * f);
              }
              hi[e] = h4;
              lo[e] = l4;
            }
            const uint32_t a = qrow + ((((uint32_t)c) ^ (ct & 7)) << 4);
            sts128(a, hi[0], hi[1], hi[2], hi[3]);
            sts128(a + kQBox, lo[0], lo[1], lo[2], lo[3]);
          }
          qinv[((qitems - 1) & 3) * 128 + ct] = xinv;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&B.qs_full[(qitems - 1) & 3]);
          if (even) mbar_arrive(&B.q16_full[qb]);
          else mbar_arrive_cluster_smem(q16_even[qb]);
        }
        for (int kt = 0; kt < it.nmax; ++kt, ++tiles) {
          const int st8 = tiles % L::kRing8;
          const uint32_t ph8 = (tiles / L::kRing8) & 1;
          // ---- V: key ct, this CTA's 64 dims
          const int vb = tiles % L::kRingV;
          if (ok) ok = mbar_wait_warp(&B.v8_full[st8], ph8, p.status);
          if (tiles >= (uint32_t)L::kRingV) {
            const uint32_t g2 = tiles - L::kRingV;  // P.V(tiles - 3) done: the stage is free
            if (ok) ok = mbar_wait_warp(&B.o_done[g2 % kNumS], (g2 / kNumS) & 1, p.status);
          }
          {
            const int key = ct, sw = key & 7, sw8 = (key >> 1) & 3;  // 64-byte rows, 64-byte swizzle
            const uint32_t src8 = smem_u32(smem + L::kV8 + st8 * kV8Bytes) + key * 64;
            const uint32_t dst = smem_u32(smem + L::kV + vb * kVBytes) + key * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) {  // dims 16 c .. + 15 of the half
              uint4 lo, hi;
              e4m3x16_to_f16(lds128(src8 + ((((uint32_t)c) ^ sw8) << 4)), lo, hi);
              sts128(dst + ((((uint32_t)(2 * c)) ^ sw) << 4), lo.x, lo.y, lo.z, lo.w);
              sts128(dst + ((((uint32_t)(2 * c + 1)) ^ sw) << 4), hi.x, hi.y, hi.z, hi.w);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&B.v16_full[vb]);
            mbar_arrive(&B.v8_empty[st8]);
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    // two threads per row of tile `rank`: warps w and w + 4 share TMEM lanes
    // 32 (w % 4) .. +31; half 0 takes columns 0-63, half 1 columns 64-127
    const int quarter = warp & 3;
    const int half = (warp - kSoftWarp0) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int t = (warp - kSoftWarp0) * 32 + lane;  // 0..255 within the group
    const int xbar = 1 + quarter;                   // named barrier of this row quarter's two warps
    const uint32_t o_cols = tmem + lane_base + kColO + half * 64;
    const uint32_t p_full_even[kNumS] = {mapa_shared(smem_u32(&B.p_full[0]), 0),
                                         mapa_shared(smem_u32(&B.p_full[1]), 0),
                                         mapa_shared(smem_u32(&B.p_full[2]), 0)};
    float* x_mine = xch + half * 128 + row;
    const float* x_other = xch + (1 - half) * 128 + row;
    float c = p.scale_log2;  // FP8: times the item's k_scale
    if (blockIdx.x == 0 && warp == kSoftWarp0 && p.status) {
      int sum = 0;
      for (int e = lane; e < p.B; e += 32) sum += max(__ldg(p.chunk_lens + e), 0);
#pragma unroll
      for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (lane == 0 && sum != p.T) atomicOr(p.status, PA_STATUS_BAD_TOKENS);
    }
    // After a wait gives up (PA_STATUS_TIMEOUT) the warps skip every later
    // wait but still walk all items and steps, so the two warps of a row
    // quarter keep meeting at the same named barriers and reach the end.
    uint32_t g = 0;       // steps so far (all items)
    uint32_t qitems = 0;  // items with key tiles so far
    bool ok = true;
    Item it;
    for (int r = 0; src.get(p, r, it); ++r) {
      const bool reporter = even && t == 0 && it.pair == 0 && it.g == 0 && p.status;
      const int nrows = it.nrows[rank];
      const int64_t tok = (int64_t)it.tok0 + rank * 128 + row;
      const bool row_valid = row < nrows;
      const bool row_out = row_valid && tok >= 0 && tok < p.T;
      uint8_t* dst = reinterpret_cast<uint8_t*>(p.out) +
                     ((tok * p.Hq + it.g) * kHeadDim + half * 64) * (p.out_f32 ? 4 : 2);
      if (it.nmax == 0) {
        // lengths invalid: zero rows
        if (!it.len_ok && reporter) atomicOr(p.status, PA_STATUS_BAD_LENGTH);
        if (row_out)
          for (int cc = 0; cc < (p.out_f32 ? 16 : 8); ++cc)
            reinterpret_cast<uint4*>(dst)[cc] = make_uint4(0, 0, 0, 0);
        continue;
      }
      if constexpr (FP8) {
        // the item's K scale and this row's 1 / x of the query split
        const uint32_t qs = qitems & 3;
        if (ok) ok = mbar_wait_warp(&B.qs_full[qs], (qitems >> 2) & 1, p.status);
        c = p.scale_log2 * __ldg(p.k_scale + it.h) * qinv[qs * 128 + row];
      }
      ++qitems;
      const int pos = it.prior + it.pair * 256 + (int)rank * 128 + row;  // this row's position
      const int last_page = (it.ctx - 1) / kPage;
      const int vtail = it.ctx % kPage;  // rows >= vtail of the last page are past the context
      const bool zero_tail = vtail != 0 && it.nmax - 1 == last_page;
      // block-table entries of the context: the first 32 loaded now, checked
      // after the key tiles (off the path to the first tile)
      const int used = (it.ctx + kPage - 1) / kPage;
      const int32_t* bt = p.block_table + (int64_t)it.s * p.max_pages;
      const int pg_first = lane < used ? __ldg(bt + lane) : 0;
      float m = -INFINITY, l = 0.f;  // l: this half's share of the row sum
      for (int kt = 0; kt < it.nmax; ++kt, ++g) {
        if (ok) ok = mbar_wait_warp(&B.s_full[g % kNumS], (g / kNumS) & 1, p.status);
        tc_fence_after();
        const uint32_t s_cols = tmem + lane_base + kColS + (g % kNumS) * 128 + half * 64;
        // causal mask only where the tile crosses pos: masked scores take no part
        const int key0 = kt * kPage + half * 64;
        const int nvis = row_valid ? min(max(pos - key0 + 1, 0), 64) : 0;  // visible keys of this half
        // warp-uniform choices: the TMEM loads and stores below are .sync.aligned
        // (both warps of a quarter hold the same rows, so they choose alike)
        const bool diag = __any_sync(0xffffffffu, nvis < 64);
        const float2 c2 = make_float2(c, c);
        // BF16 P: the row's first key tile takes the exact max of c * s over the
        // visible keys as the reference, so the largest weight is exactly 1 (with
        // few keys per row its rounding error would dominate).  The FP8 cache's
        // F16 P is 8x finer: its first tile runs against 0 (below).
        if (!FP8 && __any_sync(0xffffffffu, m == -INFINITY)) {
          float mx = -INFINITY;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t sr[32];
            tmem_ld32(s_cols + cc * 32, sr);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const float v = __uint_as_float(sr[e]) * c;
              mx = fmaxf(mx, cc * 32 + e < nvis ? v : -INFINITY);
            }
          }
          *x_mine = mx;
          named_bar_sync(xbar, 64);
          mx = fmaxf(mx, *x_other);
          named_bar_sync(xbar, 64);  // the slot is free for the next exchange
          if (m == -INFINITY) m = mx;
        }
        // One pass, speculatively against the running reference m: p = 2^(c s - m),
        // tracking the largest exponent.  The reference moves (and the tile is
        // redone) only when some visible score of the row exceeds it by more than 2^8.
        float alpha = 1.f;
        bool rescale = false;
        uint32_t pw[32];  // P as BF16 pairs (this half's 64 keys)
        float2 sum2;
        auto pass = [&](float m_ref, auto masked) -> float {
          const float2 nm2 = make_float2(-m_ref, -m_ref);
          float dmax = -INFINITY;
          sum2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
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
              // P as the MMA's operand type (F16 with the FP8 cache's F16 V)
              const float p0 = fast_exp2(d2.x), p1 = fast_exp2(d2.y);
              const uint32_t w = FP8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
              pw[cc * 16 + e] = w;
              // the normaliser adds the weights as rounded, as the MMA uses them
              sum2 = __fadd2_rn(sum2, FP8 ? f16x2_to_float2(w) : bf16x2_to_float2(w));
            }
          }
          return dmax;
        };
        const float m_use = m == -INFINITY ? 0.f : m;  // nothing visible yet: every p = 0
        // FP8 cache, the row's first key tile (no reference yet): against 0, kept
        // when the half's largest visible weight lies in [1, 2^8]; otherwise the
        // row takes its exact max as the reference and redoes the tile
        const bool first = FP8 && m == -INFINITY;  // the same for every row of the warp
        float dmax = diag ? pass(m_use, std::true_type{}) : pass(m_use, std::false_type{});
        const bool trig = dmax > kRescaleThreshold || (first && nvis > 0 && !(dmax >= 0.f));
        if (named_bar_red_or(trig, xbar, 64)) {
          // rare: the row's reference moves up to the larger of the two halves'
          // maxima, and both halves redo the tile against it
          *x_mine = dmax;
          named_bar_sync(xbar, 64);
          dmax = fmaxf(dmax, *x_other);
          float shift = dmax > kRescaleThreshold ? dmax : 0.f;
          if (first) shift = dmax == -INFINITY ? 0.f : dmax;
          const float m_new = m_use + shift;
          if (shift != 0.f) {
            if (!first) {
              alpha = fast_exp2(-shift);
              rescale = true;
            }
            m = m_new;
          }
          // warp-uniform: the pass holds .sync.aligned tensor-memory loads (a
          // lane whose row keeps its reference recomputes the same weights)
          if (__any_sync(0xffffffffu, shift != 0.f)) {
            if (diag) pass(m_new, std::true_type{}); else pass(m_new, std::false_type{});
          }
        }
        if (m == -INFINITY) m = m_use;
        l = l * alpha + (sum2.x + sum2.y);
        // P over this half's scores (all of them read above)
        tmem_st32(s_cols, pw);
        // warp-uniform: lanes that need no rescale take alpha = 1 (exact)
        if (__any_sync(0xffffffffu, rescale) && kt > 0) {
          // O must hold every earlier step: P.V(g - 1) done.  (S(g) complete
          // means P.V(g - 3) is, so this barrier is at most one phase behind.)
          const uint32_t g1 = g - 1;
          if (ok) ok = mbar_wait_warp(&B.o_done[g1 % kNumS], (g1 / kNumS) & 1, p.status);
          tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t orow[32];
            tmem_ld32(o_cols + cc * 32, orow);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) orow[e] = __float_as_uint(__uint_as_float(orow[e]) * alpha);
            tmem_st32(o_cols + cc * 32, orow);
          }
        }
        // this CTA's V half of the step: landed, and zeroed past the context
        const int vs = g % L::kRingV;
        if (ok) ok = mbar_wait_warp(FP8 ? &B.v16_full[vs] : &B.v_full[vs], (g / L::kRingV) & 1,
                                    p.status);
        if (zero_tail && kt == it.nmax - 1) {
          const int rr = vtail + (t >> 1);
          if (rr < kPage) {
            const uint32_t vb = smem_u32(smem + L::kV + vs * kVBytes) + rr * 128 + (t & 1) * 64;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) sts128(vb + ch * 16, 0u, 0u, 0u, 0u);
          }
        }
        fence_proxy_async_smem();
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (even) mbar_arrive(&B.p_full[g % kNumS]);
          else mbar_arrive_cluster_smem(p_full_even[g % kNumS]);
        }
      }
      bool pg_bad = pg_first < 0 || pg_first >= p.num_pages;
      for (int e = lane + 32; e < used; e += 32) {
        const int pg = __ldg(bt + e);
        pg_bad |= (pg < 0 || pg >= p.num_pages);
      }
      const bool bad = __any_sync(0xffffffffu, pg_bad);
      if (bad && reporter) atomicOr(p.status, PA_STATUS_BAD_PAGE);
      // ---- epilogue: O / l for this half-row, once the item's last P.V is done
      named_bar_sync(xbar, 64);  // the partner's last reads of the slot are done
      *x_mine = l;
      named_bar_sync(xbar, 64);
      const float lrow = l + *x_other;
      named_bar_sync(xbar, 64);  // the slot is free for the next item
      const uint32_t gl = g - 1;
      if (ok) ok = mbar_wait_warp(&B.o_done[gl % kNumS], (gl / kNumS) & 1, p.status);
      tc_fence_after();
      // FP8: the V codes' scale comes in here
      const float inv = lrow > 0.f ? (FP8 ? __ldg(p.v_scale + it.h) : 1.f) / lrow : 0.f;
      // an invalid sequence may have read a substitute page: select zeros
      const uint32_t keep = bad ? 0u : 0xffffffffu;
      // a full tile of BF16 rows: staged and stored by TMA (uniform over the CTA)
      const int64_t tile0 = (int64_t)it.tok0 + rank * 128;
      if (!p.out_f32 && nrows == 128 && tile0 + 128 <= p.T) {
        // the previous tile's store has finished reading the staging area
        if (t == 0) bulk_wait_read_all();
        named_bar_sync(5, 32 * kSoftmaxWarps);
        const uint32_t o_row = smem_u32(smem + L::kOut) + half * kOutBox + row * 128;
        const uint32_t sw = (uint32_t)(row & 7);
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t o0[32];
          tmem_ld32(o_cols + cc * 32, o0);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float* f = reinterpret_cast<const float*>(o0) + 8 * e;
            sts128(o_row + (((uint32_t)(cc * 4 + e) ^ sw) << 4),
                   pack_bf16x2(f[0] * inv, f[1] * inv) & keep, pack_bf16x2(f[2] * inv, f[3] * inv) & keep,
                   pack_bf16x2(f[4] * inv, f[5] * inv) & keep, pack_bf16x2(f[6] * inv, f[7] * inv) & keep);
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(5, 32 * kSoftmaxWarps);
        if (t == 0) {
          tma_store_3d(&tm_o, smem + L::kOut, 0, it.g, (int32_t)tile0);
          tma_store_3d(&tm_o, smem + L::kOut + kOutBox, 64, it.g, (int32_t)tile0);
          bulk_commit_group();
        }
        continue;
      }
      for (int cc = 0; cc < 2; ++cc) {
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
    }
  }
  // the output stores complete before the CTA exits
  if (warp == kSoftWarp0 && lane == 0) bulk_wait_all();
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

}  // namespace

namespace {

// CTA pairs that can be resident at once for one variant (cached per device).
template <bool FP8>
cudaError_t pairs_of(int num_sms, int* pairs) {
  using L = Lay<FP8>;
  static int pairs_cache[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && pairs_cache[dev] > 0) {
    *pairs = pairs_cache[dev];
    return cudaSuccess;
  }
  if ((e = cudaFuncSetAttribute(prefill_kernel<FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                L::kSmem)) != cudaSuccess)
    return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(L::kThreads);
  cfg.dynamicSmemBytes = L::kSmem;
  cfg.gridDim = dim3(2 * (num_sms / 2 > 0 ? num_sms / 2 : 1));
  int n = 0;
  if ((e = cudaOccupancyMaxActiveClusters(&n, prefill_kernel<FP8>, &cfg)) != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  if (dev >= 0 && dev < 64) pairs_cache[dev] = n;
  *pairs = n;
  return cudaSuccess;
}

template <bool FP8>
cudaError_t launch_variant(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                           const CUtensorMap& tm_q, const CUtensorMap& tm_o,
                           const PrefillParams& p, int num_sms, cudaStream_t stream) {
  using L = Lay<FP8>;
  // persistent: one CTA per SM, as many pairs as can be resident at once
  // (tensor memory and shared memory are sized for one CTA per SM)
  int pairs = 0;
  cudaError_t e = pairs_of<FP8>(num_sms, &pairs);
  if (e != cudaSuccess) return e;
  const int64_t max_items = ((int64_t)p.T / 256 + p.B) * p.Hq;
  const int grid_pairs = (int)(max_items < pairs ? max_items : pairs);
  if (grid_pairs < 1) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cfg.blockDim = dim3(L::kThreads);
  cfg.dynamicSmemBytes = L::kSmem;
  cfg.stream = stream;
  cfg.gridDim = dim3(2 * grid_pairs);
  e = cudaLaunchKernelEx(&cfg, prefill_kernel<FP8>, tm_k, tm_v, tm_q, tm_o, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t prefill_pairs(int num_sms, int* pairs) { return pairs_of<false>(num_sms, pairs); }

cudaError_t launch_prefill(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                           const CUtensorMap& tm_q, const CUtensorMap& tm_o,
                           const PrefillParams& p, int num_sms, cudaStream_t stream) {
  return p.k_scale ? launch_variant<true>(tm_k, tm_v, tm_q, tm_o, p, num_sms, stream)
                   : launch_variant<false>(tm_k, tm_v, tm_q, tm_o, p, num_sms, stream);
}

}  // namespace pa
