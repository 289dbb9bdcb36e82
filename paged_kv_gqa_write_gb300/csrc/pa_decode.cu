// pa_decode.cu -- paged GQA decode attention, flash-decoding split-K, with the
// two contractions on the 5th-generation tensor cores; one kernel template for
// a bf16 or an FP8 (e4m3) cache and one or several new tokens per sequence.
//
// Computes, for every sequence s and query head g (KV head h = g / G):
//   out[s][g] = softmax(scale * q[s][g] . K_t) V_t over t < context_lens[s],
// with K_t / V_t gathered through the block table ("Qwen3-14B" pypto-lib doc,
// "decode_fwd": paged attention after the KV cache write, vLLM ABI with flat
// [page, token, kv_head, dim] K/V; "Qwen 3" TensorSharp doc, section 11: K/V
// gathered per sequence from the block tables and sequence lengths).
//
// Design (GB300; HBM bound: every K/V byte is read once):
//  * Persistent grid, one CTA per SM.  A work item is (split j, sequence s,
//    KV head h, token group): a contiguous range of at most `pps` pages and
//    the GC = Lg * G <= 32 (token, query head) columns of the G query heads
//    that share the KV head, for Lg of the sequence's L new tokens (L = 1:
//    the plain decode, one column per head).  With several new tokens the
//    columns of all of them share each K/V page as long as they fit, so the
//    pages are read once per KV head, not once per token.  Items are dealt round-robin;
//    split boundaries depend only on logical positions.
//  * Per page the two products are transposed so that the 128 keys (or the
//    128 head dims) fill the 128 rows of one tcgen05.mma and the columns,
//    padded to 16 or 32, are its N:
//      S^T[key][g] = K[key][:] . Q[g][:]        (A = K tile, K-major)
//      O^T[d][g]  += V[:][d] . P[g][:]          (A = V tile, MN-major)
//    so the K/V tiles are read by the tensor core straight from the TMA ring
//    (128-byte swizzle), and the FP32 pipes only run the softmax.
//  * warp 0: validates each item's block-table range (the next item's
//    metadata is loaded while the current item's pages are issued), stages
//    up to four items ahead (two with 32 columns), TMA-loads each item's query rows (G heads, or a
//    3-D box of Lg tokens x G heads; rows past it stay zero) and its K/V page
//    tiles into a 3-stage ring of 64 KB (K and V complete on separate
//    mbarriers, so QK^T starts while V is in flight).
//  * warp 1: owns TMEM (S[2], O[2]) and issues the MMAs: QK^T(j + 1) before
//    P.V(j), into the other of two S buffers, so the tensor core computes the
//    next page's scores while the softmax works on this page's; P.V(j) once
//    P(j) is in its shared-memory buffer (two, by page parity).  FP8 cache:
//    warp 1 issues QK^T only and warp 14 P.V, each on its own thread.
//  * warps 2-5, one thread per key: tcgen05.ld of the key's scores, online
//    softmax in the log2 domain with a per-head reference max shared by the
//    CTA.  The reference only moves when some score exceeds it by more than
//    2^8 (a vote exchanged among the four warps decides), which rescales O in
//    TMEM after the previous P.V; the first page of an item takes the exact
//    max.  The warps agree through a small shared-memory exchange on
//    mbarriers (bounded waits, no bar.sync).  P is rounded to BF16 (F16 for
//    the FP8 cache) and written transposed into a K-major operand; the row
//    sums accumulate the rounded values, so the normalisation matches the
//    weights the MMA used.  V rows past the context in the last page are
//    zeroed before P.V reads them (P is 0 there, but 0 * NaN is NaN).
//  * warps 6-9, one thread per head dim: the epilogue of the previous item
//    (O / l from TMEM, double-buffered) overlaps the next item's pages; it
//    writes `out` (one split) or normalised partials (o, lse) for the combine.
//  * FP8 cache: TMA lands e4m3 pages.  QK^T runs on the e4m3 K page itself
//    (kind::f8f6f4, K-major): the TMA warp splits each query row into two
//    e4m3 rows whose sum is the row (times a power of two), so S^T has a hi
//    and a lo column per query column, which the softmax adds.  Converter
//    warps rewrite V as F16 into shared memory for P.V (kind::f16).
//  * In-kernel prologue (pa_decode_prologue; "Qwen3-14B", decode_fwd: the
//    attention kernel there runs the RoPE/QKV step as its phase 0): warp 10
//    walks the same items as the TMA warp, builds each item's query operand
//    from the fused QKV row (per-head RMSNorm, NeoX RoPE, the Q scale) and
//    stores the new token's K/V row into its slot ahead of the page load that
//    reads it, so the TMA warp's page loads never wait for that arithmetic.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "pa_launch.cuh"

namespace pa {
namespace {

constexpr int kTmaWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kSoftWarp0 = 2;  // warps 2-5: softmax, one thread per key
constexpr int kEpiWarp0 = 6;   // warps 6-9: epilogue, one thread per head dim
constexpr int kConvWarp0 = 10; // FP8 cache: warps 10-13 convert V, one thread per key row
constexpr int kProWarp = 10;   // in-kernel prologue (bf16 cache only): builds the query operands
constexpr int kBalMaxSeqs = PA_BALANCED_MAX_SEQS;  // page-balanced schedule: sequences
constexpr int kBox = 64 * 2 * kPage;       // 64 dims x 128 tokens of bf16 = 16 KB
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.69314718055994530942f;

// Item record in shared memory, written by the TMA warp, read by every role.
enum : int {
  kICtx = 0,   // context length of the sequence
  kIPg0 = 1,   // first page of the item
  kIPg1 = 2,   // end page (== kIPg0 when the item has no pages to read)
  kIFlag = 3,  // 0 ok, 1 invalid block-table entry, 2 invalid context length
  kISeq = 4,   // sequence
  kIUnit = 5,  // KV head * NT + token group
  kIDest = 6,  // -1: out; else the partial record (split index, or 2 * CTA + cut side)
  kIDone = 7,  // no more items
  kIQInv = 8,  // FP8: 1 / x (float bits), x the power of two the query rows were scaled by
  kInfoInts = 10
};

// Shared memory (offsets from a 1024-aligned base).  BF16 cache: a 3-stage
// ring of K/V operand pages loaded by TMA.  FP8 cache: a 4-stage ring of e4m3
// pages (32 KB each) loaded by TMA; QK^T reads the K tile there, and the
// converter warps rewrite each page's V as F16 into a 2-stage shared-memory
// ring (the tensor core reads F16; every e4m3 value is exact in it).
constexpr int kBox8 = 128 * kPage;         // 128 one-byte dims x 128 tokens = 16 KB
constexpr uint32_t pow2_cols(uint32_t n) { return n <= 32 ? 32 : n <= 64 ? 64 : n <= 128 ? 128 : 256; }
template <bool FP8, int NH = 16>
struct Layout {
  // MMA N: the item's (token, query head) columns, padded to 16 or 32
  static constexpr int kN = NH > 16 ? 32 : 16;
  // QK^T's N: FP8 doubles the query columns (hi rows 0 .. NH - 1, lo rows
  // NH .. 2 NH - 1 of the e4m3 query operand)
  static constexpr int kNS = FP8 ? (2 * NH > kN ? 2 * NH : kN) : kN;
  static constexpr int kAtom = kN * 128;     // kN rows x 128 bytes
  static constexpr int kOpBytes = 2 * kAtom; // Q or P operand: two 64-element atoms
  static_assert(kNS * 128 <= kOpBytes, "the e4m3 query operand fits the query slot");
  // item slots: how far the TMA warp runs ahead (two with the wide operands,
  // which the shared-memory budget allows no more of)
  static constexpr int kSlots = kN == 32 ? 2 : 4;
  // tensor-memory columns: S^T[2] (kNS each) and O^T[2] (kN each)
  static constexpr uint32_t kColS = 0, kColO = 2 * kNS;
  // operand stages: bf16 K lo, K hi, V lo, V hi; FP8 V lo, V hi as F16
  static constexpr int kStages = FP8 ? 2 : 3;
  static constexpr int kStageBytes = FP8 ? 2 * kBox : 4 * kBox;
  static constexpr int kStages8 = FP8 ? 4 : 0;  // e4m3 pages (K, V)
  // V converter warps, one thread per key row
  static constexpr int kConvWarps = FP8 ? 4 : 0;
  // FP8: P.V has an issuing thread of its own (warp 14), QK^T stays on warp 1
  static constexpr bool kSplitIssue = FP8;
  static constexpr int kPvWarp = 10 + kConvWarps;
  static constexpr int kThreads = (10 + kConvWarps + (kSplitIssue ? 1 : 0)) * 32;
  static constexpr int kRing = 0;
  static constexpr int kRing8 = kRing + kStages * kStageBytes;
  static constexpr uint32_t kTmemCols = pow2_cols(2 * kNS + 2 * kN);
  static constexpr int kQ = kRing8 + kStages8 * 2 * kBox8;  // [kSlots] query operands
  static constexpr int kP = kQ + kSlots * kOpBytes;         // P operands [2]
  static constexpr int kX = kP + 2 * kOpBytes;              // float [2][4][kN]: softmax exchange
  static constexpr int kML = kX + 2 * 4 * kN * 4;           // float [2][kN][2]: (m, l) per O
  static constexpr int kInfo = kML + 2 * kN * 2 * 4;        // int [kSlots][kInfoInts]: item records
  static constexpr int kBars = kInfo + kSlots * kInfoInts * 4;
  static constexpr int kNumBars =
      3 * kStages + 3 * kStages8 + 2 * kSlots + 2 * 2 + 2 + 4 * 2 + 1 +
      (kN == 32 ? 2 : 0) +  // 32 columns: a second pair of exchange slots
      kSlots;               // the in-kernel prologue's K/V-row barriers
  // in-kernel prologue: the RoPE tables (64 double frequencies, 64 + 64 float
  // turn rates), staged from the kernel parameters
  static constexpr int kRope = kBars + kNumBars * 8 + 16;
  static constexpr int kRopeBytes = (!FP8 && NH <= 16) ? 64 * 8 + 2 * 64 * 4 : 0;
  static constexpr int kSmem = kRope + kRopeBytes + 1024;  // + room to align the base
};
constexpr int kSmemLimit = 232448;
static_assert(Layout<false>::kSmem <= kSmemLimit, "decode shared memory exceeds the limit");
static_assert(Layout<true>::kSmem <= kSmemLimit, "FP8 decode shared memory exceeds the limit");
static_assert(Layout<false, 32>::kSmem <= kSmemLimit, "wide decode shared memory exceeds the limit");
static_assert(Layout<true, 32>::kSmem <= kSmemLimit, "wide FP8 decode shared memory exceeds the limit");

// TMEM loads and stores of one lane's kN columns
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 32) tmem_ld32(taddr, r); else tmem_ld16(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[N]) {
  if constexpr (N == 32) tmem_st32(taddr, r); else tmem_st16(taddr, r);
}

struct Bars {
  uint64_t* k_full;    // [kStages] operand page: K landed (bf16)
  uint64_t* v_full;    // [kStages] V ready (TMA, or the FP8 converters)
  uint64_t* kv_empty;  // [kStages] P.V of the page done
  uint64_t* k8_full;   // [kStages8] FP8: e4m3 K tile landed
  uint64_t* v8_full;   // [kStages8] FP8: e4m3 V tile landed
  uint64_t* kv8_empty; // [kStages8] FP8: QK^T done with K and the converters with V
  uint64_t* q_full;    // [kSlots] item slot staged (info + query operand)
  uint64_t* q_empty;   // [kSlots] item slot read by every role, query operand used
  uint64_t* s_full;    // [2] S^T of a page (by page parity)
  uint64_t* p_full;    // [2] P of a page
  uint64_t* pv_done;   // [2] P.V of a page done (by page parity): its P buffer is free,
                       // and the softmax's O rescale of the next page may run
  uint64_t* o_full;    // [2] last P.V of the item done
  uint64_t* o_free;    // [2] epilogue read O and (m, l)
  uint64_t* ml_full;   // [2] (m, l) of the item published
  uint64_t* x_full;    // [2] softmax-warp exchange slots (one arrival per warp)
  uint64_t* mma_done;  // drain at exit
  uint64_t* kv_ready;  // [kSlots] in-kernel prologue: the item's new K/V row stored (or none)
};

// A work item: pages [pg0, pg1) of unit (s, unit) whose result goes to `dest`.
struct Work {
  int s, unit, ctx, pg0, pg1, dest;
};

__device__ __forceinline__ bool ctx_ok(int ctx, const DecodeParams& p) {
  return ctx >= 0 && ctx <= p.max_pages * kPage;
}

__device__ __forceinline__ int pages_of(int ctx, const DecodeParams& p) {
  return ctx_ok(ctx, p) ? (ctx + kPage - 1) / kPage : 0;
}

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

// Columns of work unit `unit` (KV head x token group): the group's tokens
// (the last group may hold fewer) times the query heads per KV head.
__device__ __forceinline__ int unit_columns(const DecodeParams& p, int unit) {
  const int t0 = (unit % p.NT) * p.Lg;
  return min(p.Lg, p.L - t0) * p.G;
}

// Instruction descriptor of tcgen05.mma kind::f8f6f4 with E4M3 A and B (format
// code 0), both K-major, FP32 accumulate, an M x N tile.
__host__ __device__ constexpr uint32_t umma_idesc_e4m3(int M, int N) {
  return (1u << 4)                            // D format: F32
         | ((uint32_t)(N >> 3) << 17)         // N / 8
         | ((uint32_t)(M >> 4) << 24);        // M / 16
}

// D[tmem] (+)= A[smem] * B[smem] over 32 e4m3 elements of K, issued by one thread.
__device__ __forceinline__ void umma_e4m3_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 16 columns of one lane as two 8-column accesses (any 8-column boundary)
__device__ __forceinline__ void tmem_ld8x2(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%16];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8, %9, %10, %11, %12, %13, %14, %15}, [%17];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr), "r"(taddr + 8));
}
__device__ __forceinline__ void tmem_st8x2(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%2, %3, %4, %5, %6, %7, %8, %9};\n\t"
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%1], {%10, %11, %12, %13, %14, %15, %16, %17};"
      ::"r"(taddr), "r"(taddr + 8),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// NH: columns the softmax and epilogue handle (8, 16 or 32, >= any item's GC).
// FP8: the cache holds e4m3 codes with per-KV-head scales.  MULTI: more than
// one new token per sequence (per-column causal masks, (token, head) columns);
// without it every column is a query head that sees the whole context.
// PRO: the decode step's prologue runs in this kernel (bf16 cache, one new
// token per sequence): the TMA warp builds each item's query operand from the
// fused QKV row (per-head RMSNorm, NeoX RoPE at the new token's position, the
// Q scale) instead of loading q, and before it loads the page that holds the
// new token it writes that token's K row (normed, rotated) and V row into the
// cache slot -- the arithmetic of pa_qk_norm_rope_write, so the same bits.
template <int NH, bool FP8, bool MULTI, bool PRO>
__device__ __forceinline__ void decode_body(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                            const CUtensorMap& tm_q, const DecodeParams& p,
                                            const DecodePrologue* pro) {
  static_assert(!PRO || (!FP8 && !MULTI), "the in-kernel prologue serves the bf16 single-token kernel");
  using Lay = Layout<FP8, NH>;
  constexpr int kConvWarps = Lay::kConvWarps;
  constexpr int kStages = Lay::kStages, kStageBytes = Lay::kStageBytes;
  constexpr int kStages8 = FP8 ? Lay::kStages8 : 1;  // (the bf16 kernel has no e4m3 ring)
  constexpr int kRing = Lay::kRing, kRing8 = Lay::kRing8, kQ = Lay::kQ, kP = Lay::kP;
  constexpr int kX = Lay::kX, kML = Lay::kML, kInfo = Lay::kInfo, kBars = Lay::kBars;
  constexpr int kNumBars = Lay::kNumBars, kThreads = Lay::kThreads;
  constexpr int kN = Lay::kN, kAtom = Lay::kAtom, kOpBytes = Lay::kOpBytes, kSlots = Lay::kSlots;
  constexpr int kNS = Lay::kNS;
  constexpr uint32_t kColS = Lay::kColS, kColO = Lay::kColO;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kBars);
  Bars B;
  B.k_full = bar;
  B.v_full = B.k_full + kStages;
  B.kv_empty = B.v_full + kStages;
  B.k8_full = B.kv_empty + kStages;
  B.v8_full = B.k8_full + Lay::kStages8;  // (none in the bf16 kernel)
  B.kv8_empty = B.v8_full + Lay::kStages8;
  B.q_full = B.kv8_empty + Lay::kStages8;
  B.q_empty = B.q_full + kSlots;
  B.s_full = B.q_empty + kSlots;
  B.p_full = B.s_full + 2;
  B.pv_done = B.p_full + 2;
  B.o_full = B.pv_done + 2;
  B.o_free = B.o_full + 2;
  B.ml_full = B.o_free + 2;
  B.x_full = B.ml_full + 2;
  B.mma_done = B.x_full + (kN == 32 ? 4 : 2);
  B.kv_ready = B.mma_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBars + kNumBars * 8);
  int* info = reinterpret_cast<int*>(smem + kInfo);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&B.k_full[i], 1);
      mbar_init(&B.v_full[i], FP8 ? kConvWarps : 1);  // FP8: one arrival per converter warp
      mbar_init(&B.kv_empty[i], 1);
    }
    for (int i = 0; i < Lay::kStages8; ++i) {
      mbar_init(&B.k8_full[i], 1);
      mbar_init(&B.v8_full[i], 1);
      mbar_init(&B.kv8_empty[i], kConvWarps + 1);  // + the QK^T commit
    }
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&B.q_full[i], PRO ? 2 : 1);  // PRO: the record and the query operand
      mbar_init(&B.kv_ready[i], 1);
      // the MMA issuer(s), 4 softmax warps, 4 epilogue warps (, the converter warps)
      mbar_init(&B.q_empty[i], (Lay::kSplitIssue ? 2 : 1) + 4 + 4 + kConvWarps);
    }
    // 32 columns: two groups of 128 softmax threads, each also its columns' epilogue
    constexpr uint32_t kColThreads = kN == 32 ? 256 : 128;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B.o_full[i], 1);
      mbar_init(&B.o_free[i], kColThreads);
      mbar_init(&B.ml_full[i], 1);
    }
    for (int i = 0; i < (kN == 32 ? 4 : 2); ++i) mbar_init(&B.x_full[i], 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B.s_full[i], 1);
      mbar_init(&B.p_full[i], kColThreads);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&B.pv_done[i], 1);
    mbar_init(B.mma_done, Lay::kSplitIssue ? 2 : 1);  // every issuing thread
    fence_mbar_init();
  }
  // query rows past every item's box and unused P rows read as zero: clear the
  // operands (columns past an item's GC are computed and never used)
  for (int o = threadIdx.x * 16; o < (kSlots + 2) * kOpBytes; o += kThreads * 16)
    sts128(smem_u32(smem + kQ + o), 0u, 0u, 0u, 0u);
  if constexpr (PRO) {
    // per-lane reads of the parameter block diverge; shared memory does not
    double* rope_f = reinterpret_cast<double*>(smem + Lay::kRope);
    float* rope_t = reinterpret_cast<float*>(smem + Lay::kRope + 64 * 8);
    if (threadIdx.x < 64) {
      rope_f[threadIdx.x] = pro->freq[threadIdx.x];
      rope_t[threadIdx.x] = pro->turn_hi[threadIdx.x];
      rope_t[64 + threadIdx.x] = pro->turn_lo[threadIdx.x];
    }
  }
  fence_proxy_async_smem();
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, Lay::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Launched as a programmatic dependent of the kernel before it on the
  // stream (a KV write, say): everything above touches only this CTA's shared
  // and tensor memory; every global access comes after that kernel has
  // completed and its writes are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // a combine launched as a programmatic dependent may start its prologue now;
  // it reads partials only after this grid has completed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == kTmaWarp || (PRO && warp == kProWarp)) {
    // ------------------------------------------------------------ TMA producer
    // (PRO: and the prologue warp, which walks the same items: it builds each
    // item's query operand and stores the new token's K/V row, so that the
    // TMA warp's page loads never wait for that arithmetic)
    const bool tma = warp == kTmaWarp;
    if (tma && lane == 0) {
      prefetch_tensor_map(&tm_k);
      prefetch_tensor_map(&tm_v);
      if (!PRO) prefetch_tensor_map(&tm_q);
    }
    const uint64_t pol = l2_policy_evict_first();
    // PRO: lane li of each half-warp holds the norm weights of values
    // 4 li .. 4 li + 3 and 64 + 4 li .. (the layout of the prologue's compute lanes)
    const int pli = lane & 15;
    float4 pwq_lo{}, pwq_hi{}, pwk_lo{}, pwk_hi{};
    float pgmax = 0.f;
    float pth[4] = {}, ptl[4] = {};  // this lane's four pairs' turn rates (hi + lo)
    double pfq[4] = {};               // ... and radians per position
    if (PRO && !tma) {
      const double* rope_f = reinterpret_cast<const double*>(smem + Lay::kRope);
      const float* rope_t = reinterpret_cast<const float*>(smem + Lay::kRope + 64 * 8);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        pth[j] = rope_t[4 * pli + j];
        ptl[j] = rope_t[64 + 4 * pli + j];
        pfq[j] = rope_f[4 * pli + j];
      }
      pwq_lo = __ldg(reinterpret_cast<const float4*>(pro->wq + 4 * pli));
      pwq_hi = __ldg(reinterpret_cast<const float4*>(pro->wq + 4 * pli + 64));
      pwk_lo = __ldg(reinterpret_cast<const float4*>(pro->wk + 4 * pli));
      pwk_hi = __ldg(reinterpret_cast<const float4*>(pro->wk + 4 * pli + 64));
      pgmax = fmaxf(rope_t[0], rope_t[63]);  // the frequencies are monotone
    }
    // ---- work generator (warp-uniform state).  Fixed splits: items
    // i = blockIdx.x + k * gridDim.x of (split, sequence, unit).  Page-balanced:
    // the CTAs form groups of UPS (one CTA per unit = KV head x head group);
    // the sequences' pages laid end to end (n_s pages for sequence s, W in
    // total) are divided evenly among the groups, and the CTA with unit j of a
    // group takes unit j of every sequence in the group's range [lo, hi) --
    // so the CTAs of a group read the same pages at about the same time.  A
    // sequence cut by lo or hi leaves partial records for the balanced
    // combine; an empty sequence (or one with an invalid length) belongs to
    // the group whose range holds its position (the last group for W).
    const int UPS = p.Hkv * p.NT;  // units per sequence
    int gi = blockIdx.x;           // fixed: next item index
    int bs = p.B, bn = 0, bctx = 0;  // balanced: sequence, its pages, its context length
    int64_t bP = 0, lo = 0, hi = 0, W = 0;
    const int ngroups = gridDim.x / UPS, grp = blockIdx.x / UPS, unit_j = blockIdx.x % UPS;
    int cbase = -64, cval = 0;     // 32 context lengths starting at cbase (lane's in cval)
    const bool last_grp = grp == ngroups - 1;
    auto ctx_at = [&](int sq) -> int {
      if (sq < cbase || sq >= cbase + 32) {
        cbase = sq;
        cval = cbase + lane < p.B ? (MULTI ? seq_ctx(p.context_lens, cbase + lane, p.L)
                                           : __ldg(p.context_lens + cbase + lane))
                                  : 0;
      }
      return __shfl_sync(0xffffffffu, cval, sq - cbase);
    };
    if (p.balanced && grp < ngroups) {
      // lane l holds the page counts of sequences 16l .. 16l+15 (B <= 512;
      // the host guarantees W < 2^31).  Loads of a clamped index are
      // unconditional, so they issue together.
      constexpr int R = kBalMaxSeqs / 32;
      int np[R];
#pragma unroll
      for (int r = 0; r < R; ++r)
        np[r] = MULTI ? seq_ctx(p.context_lens, min(lane * R + r, p.B - 1), p.L)
                      : __ldg(p.context_lens + min(lane * R + r, p.B - 1));
      int lsum = 0;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        np[r] = lane * R + r < p.B ? pages_of(np[r], p) : 0;
        lsum += np[r];
      }
      int incl = lsum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      W = __shfl_sync(0xffffffffu, incl, 31);
      lo = W * grp / ngroups;
      hi = W * (grp + 1) / ngroups;
      // first sequence the group touches: it reaches past lo, or it is empty
      // and sits at or after lo
      int start = incl - lsum, hit_r = -1, hit_start = 0;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const bool hit = lane * R + r < p.B &&
                         (start + np[r] > lo || (np[r] == 0 && start >= lo));
        if (hit && hit_r < 0) {
          hit_r = r;
          hit_start = start;
        }
        start += np[r];
      }
      const unsigned m = __ballot_sync(0xffffffffu, hit_r >= 0);
      if (m) {
        const int f = __ffs(m) - 1;
        bs = f * R + __shfl_sync(0xffffffffu, hit_r, f);
        bP = __shfl_sync(0xffffffffu, hit_start, f);
        bctx = ctx_at(bs);
        bn = pages_of(bctx, p);
      }
    }
    auto gen_next = [&](Work& w) -> bool {
      if (!p.balanced) {
        if (gi >= p.num_items) return false;
        const int U = p.B * UPS;
        const int jsp = gi / U, u = gi - jsp * U;
        w.s = u / UPS;
        w.unit = u - w.s * UPS;
        w.ctx = MULTI ? seq_ctx(p.context_lens, w.s, p.L) : __ldg(p.context_lens + w.s);
        w.pg0 = jsp * p.pps;
        w.pg1 = max(w.pg0, min(pages_of(w.ctx, p), w.pg0 + p.pps));
        w.dest = p.S == 1 ? -1 : jsp;
        gi += gridDim.x;
        return true;
      }
      if (grp >= ngroups || bs >= p.B) return false;
      if (bn == 0) {
        if (bP >= hi && !(last_grp && bP == W)) {
          bs = p.B;
          return false;
        }
        w.pg0 = 0;
        w.pg1 = 0;
        w.dest = -1;
      } else {
        if (bP >= hi || lo >= hi) {  // past the range, or an empty range
          bs = p.B;
          return false;
        }
        const int64_t a = max(bP, lo), b = min(bP + bn, hi);
        w.pg0 = (int)(a - bP);
        w.pg1 = (int)(b - bP);
        w.dest = (a == bP && b == bP + bn) ? -1 : 2 * (int)blockIdx.x + (bP <= lo ? 0 : 1);
      }
      w.s = bs;
      w.unit = unit_j;
      w.ctx = bctx;
      bP += bn;
      ++bs;
      if (bs < p.B) {
        bctx = ctx_at(bs);
        bn = pages_of(bctx, p);
      }
      return true;
    };
    // this lane's block-table entry among the first 32 pages of an item
    // (it does not wait for the context length: entries past the sequence's
    // pages are in the row and are never used)
    auto first_pid = [&](const Work& w) -> int {
      const int pg = w.pg0 + lane;
      return pg < p.max_pages ? __ldg(p.block_table + (int64_t)w.s * p.max_pages + pg) : 0;
    };
    // PRO: the fused QKV row parts an item reads (its G query heads, its K and
    // V heads), prefetched into L1 when the item is generated
    auto prefetch_row = [&](const Work& w) {
      if (PRO && !tma) {
        const uint8_t* xrow = reinterpret_cast<const uint8_t*>(pro->qkv) +
                              (int64_t)w.s * (p.Hq + 2 * p.Hkv) * (kHeadDim * 2);
        for (int i = lane; i < 2 * p.G + 4; i += 32) {
          const int64_t off = i < 2 * p.G ? (int64_t)w.unit * p.G * 256 + i * 128
                            : i < 2 * p.G + 2 ? (int64_t)(p.Hq + w.unit) * 256 + (i - 2 * p.G) * 128
                                              : (int64_t)(p.Hq + p.Hkv + w.unit) * 256 +
                                                    (i - 2 * p.G - 2) * 128;
          asm volatile("prefetch.global.L1 [%0];" ::"l"(xrow + off));
        }
      }
    };
    Work nx;
    bool have = gen_next(nx);
    int nx_pid = have ? first_pid(nx) : 0;
    if (have) prefetch_row(nx);
    uint32_t gp = 0, n = 0;
    // per item slot: parity of its last use if that use loaded a query operand, else -1
    int q_pending[kSlots];
#pragma unroll
    for (int k = 0; k < kSlots; ++k) q_pending[k] = -1;
    bool ok = true;
    for (; ok; ++n) {
      const Work w = nx;
      const int pid0 = nx_pid;
      const bool item = have;
      int flag = 0, npg = 0;
      bool pkv = false;  // PRO: this item writes the new token's K/V row
      const int slot = n % kSlots;
      float4 pc4{}, ps4{};  // PRO: cos / sin of this lane's four NeoX pairs at the new token
      if constexpr (PRO) {
        if (!tma) {
          // ---- prologue warp: the item's query operand first (it needs
          // neither the block table nor the item's validation), then the
          // validation below and the new token's K/V row
          if (!(ok = mbar_wait_warp(&B.q_empty[slot], ((n / kSlots) & 1) ^ 1, p.status))) break;
          if (item && w.pg1 > w.pg0 && w.ctx > 0 && ctx_ok(w.ctx, p)) {
            const int pos = w.ctx - 1;
            float cs[4], sn[4];
            auto angles = [&](bool fast) {
#pragma unroll
              for (int j = 0; j < 4; ++j) rope_sincos(pos, fast, pth[j], ptl[j], pfq[j], sn[j], cs[j]);
            };
            if (rope_fast(pos, pgmax)) angles(true); else angles(false);
            pc4 = make_float4(cs[0], cs[1], cs[2], cs[3]);
            ps4 = make_float4(sn[0], sn[1], sn[2], sn[3]);
            // the G query heads, a half-warp per head, into the operand in the
            // 128-byte-swizzled layout the TMA load gives (rows past G stay zero)
            const uint8_t* qrow = reinterpret_cast<const uint8_t*>(pro->qkv) +
                                  ((int64_t)w.s * (p.Hq + 2 * p.Hkv) + w.unit * p.G) * (kHeadDim * 2);
            const uint32_t qd = smem_u32(smem + kQ + slot * kOpBytes);
            constexpr int kPasses = (NH + 1) / 2;
            uint2 ra[kPasses], rb[kPasses];
#pragma unroll
            for (int m = 0; m < kPasses; ++m) {
              const int r = min(2 * m + (lane >> 4), p.G - 1);
              ra[m] = __ldg(reinterpret_cast<const uint2*>(qrow + r * (kHeadDim * 2) + 8 * pli));
              rb[m] = __ldg(reinterpret_cast<const uint2*>(qrow + r * (kHeadDim * 2) + 128 + 8 * pli));
            }
#pragma unroll
            for (int m = 0; m < kPasses; ++m) {
              if (2 * m >= p.G) break;
              const int r = 2 * m + (lane >> 4);
              float4 oa, ob;
              norm_rope_half(ra[m], rb[m], pwq_lo, pwq_hi, pc4, ps4, pro->eps, pro->q_scale, oa, ob);
              if (r < p.G) {
                const uint2 qa = float4_to_bf16x4(oa), qb = float4_to_bf16x4(ob);
                const uint32_t off =
                    r * 128 + ((((uint32_t)pli >> 1) ^ ((uint32_t)r & 7)) << 4) + (pli & 1) * 8;
                sts64(qd + off, qa.x, qa.y);
                sts64(qd + kAtom + off, qb.x, qb.y);
              }
            }
            fence_proxy_async_smem();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&B.q_full[slot]);  // the query operand is in place
        }
      }
      if (item) {
        // validate every page of the item; the next item's metadata loads
        // while this one's pages are issued
        const int32_t* bt = p.block_table + (int64_t)w.s * p.max_pages;
        bool bad = w.pg0 + lane < w.pg1 && (pid0 < 0 || pid0 >= p.num_pages);
        for (int pg = w.pg0 + 32 + lane; pg < w.pg1; pg += 32) {
          const int pid = __ldg(bt + pg);
          bad |= pid < 0 || pid >= p.num_pages;
        }
        bad = __any_sync(0xffffffffu, bad);
        flag = !ctx_ok(w.ctx, p) ? 2 : (bad ? 1 : 0);
        npg = flag ? 0 : w.pg1 - w.pg0;
        if constexpr (PRO) {
          // the new token's K/V row is written by the item that reads the page
          // holding it, once every block-table entry of the sequence is valid
          // (the prologue writes nothing for an invalid sequence); a sequence
          // without that token (length 0) is flagged as the prologue flags it
          pkv = npg > 0 && w.pg0 + npg == pages_of(w.ctx, p);
          if (pkv) {
            bool bad0 = false;
            for (int e = lane; e < w.pg0; e += 32) {
              const int pid = __ldg(bt + e);
              bad0 |= pid < 0 || pid >= p.num_pages;
            }
            pkv = !__any_sync(0xffffffffu, bad0);
          }
          if (w.ctx == 0 && w.unit == 0 && lane == 0 && p.status)
            atomicOr(p.status, PA_STATUS_BAD_LENGTH);
        }
        have = gen_next(nx);
        if (have) {
          nx_pid = first_pid(nx);
          prefetch_row(nx);
        }
      }
      if constexpr (PRO) {
        if (!tma) {
          if (pkv) {
            // the new token's K row (normed, rotated; lanes 0-15 store it) and
            // V row (copied; lanes 16-31) into its slot
            const int h = w.unit;
            const uint8_t* xrow = reinterpret_cast<const uint8_t*>(pro->qkv) +
                                  (int64_t)w.s * (p.Hq + 2 * p.Hkv) * (kHeadDim * 2);
            const uint8_t* krow = xrow + (int64_t)(p.Hq + h) * (kHeadDim * 2);
            const uint8_t* vrow = xrow + (int64_t)(p.Hq + p.Hkv + h) * (kHeadDim * 2);
            const uint2 ka = __ldg(reinterpret_cast<const uint2*>(krow + 8 * pli));
            const uint2 kb = __ldg(reinterpret_cast<const uint2*>(krow + 128 + 8 * pli));
            const uint4 vv = __ldg(reinterpret_cast<const uint4*>(vrow) + pli);
            float4 oa, ob;
            norm_rope_half(ka, kb, pwk_lo, pwk_hi, pc4, ps4, pro->eps, 1.f, oa, ob);
            const int last = npg - 1;  // the item's page holding the token
            const int pid_last = __shfl_sync(0xffffffffu, pid0, last & 31);
            const int page = last < 32 ? pid_last
                                       : __ldg(p.block_table + (int64_t)w.s * p.max_pages +
                                               w.pg0 + last);
            const int64_t slot_row = ((int64_t)page * kPage + (w.ctx - 1) % kPage) * p.Hkv + h;
            if (lane < 16) {
              uint2* kd = reinterpret_cast<uint2*>(pro->k_cache + slot_row * kHeadDim);
              kd[pli] = float4_to_bf16x4(oa);
              kd[16 + pli] = float4_to_bf16x4(ob);
            } else {
              reinterpret_cast<uint4*>(pro->v_cache + slot_row * kHeadDim)[pli] = vv;
            }
            // the stored row reaches the async proxy before the page's tensor
            // load (proxy fence in every writing lane, warp barrier, release
            // by lane 0, acquire by the TMA warp)
            fence_proxy_async_global();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&B.kv_ready[slot]);
          if (!item) break;
          continue;
        }
      }
      if (!(ok = mbar_wait_warp(&B.q_empty[slot], ((n / kSlots) & 1) ^ 1, p.status))) break;
      float q_inv = 1.f;  // FP8: 1 / x
      if constexpr (FP8) {
        if (npg > 0) {
          // QK^T reads e4m3 on both sides.  Each query row r (token r / G,
          // head r % G) times a power of two x is split into two e4m3 rows,
          // hi = e4m3(x q) at operand row r and lo = e4m3(x q - hi) at row
          // NH + r.  x brings the item's largest |q| into [128, 256), so hi
          // and lo are e4m3 values (no saturation) and hi + lo = x q exactly
          // for every element of magnitude at least 2^-2 after scaling, i.e.
          // at least 2^-10 of the largest (a bf16 value has 8 significant
          // bits, and the residual of its rounding to 4 is a multiple of its
          // last bit with at most 4 significant bits); smaller ones are off
          // by at most 2^-10 / x.
          const uint32_t qd = smem_u32(smem + kQ + slot * kOpBytes);
          const int qh = (w.unit / p.NT) * p.G;
          const int64_t qt = (int64_t)w.s * p.L + (w.unit % p.NT) * p.Lg;
          const int64_t T = (int64_t)p.B * p.L;
          const int rows = p.Lg * p.G;
          auto q_chunk = [&](int r, int k) -> uint4 {  // bf16 dims 8k .. 8k + 7 of row r
            const int64_t tok = qt + r / p.G;
            return tok < T ? __ldg(reinterpret_cast<const uint4*>(
                                       p.q + (tok * p.Hq + qh + r % p.G) * kHeadDim) + k)
                           : make_uint4(0u, 0u, 0u, 0u);
          };
          // the largest magnitude (bf16 bits: the magnitude order is the
          // integer order; above 0x7f80: inf or NaN)
          uint32_t amax = 0;
          for (int i = lane; i < rows * 16; i += 32) {
            const uint4 v = q_chunk(i >> 4, i & 15);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              amax = max(amax, max(wv[e] & 0x7fffu, (wv[e] >> 16) & 0x7fffu));
          }
          amax = __reduce_max_sync(0xffffffffu, amax);
          float x;
          if (amax >= 0x7f80u) {
            // inf or NaN in q: flagged, and the item's scores become NaN
            x = __uint_as_float(0x7fc00000u);
            if (lane == 0 && p.status) atomicOr(p.status, PA_STATUS_Q_RANGE);
          } else {
            // largest = 1.f x 2^(be - 127); x = 2^(134 - be), kept a normal float
            const int be = (int)(amax >> 7);
            const int sx = min(134 - be, 126);
            x = __uint_as_float((uint32_t)(127 + sx) << 23);
            q_inv = __uint_as_float((uint32_t)(127 - sx) << 23);
          }
          for (int i = lane; i < rows * 8; i += 32) {
            const int r = i >> 3, k = i & 7;  // dims 16k .. 16k + 15
            const uint4 va = q_chunk(r, 2 * k), vb = q_chunk(r, 2 * k + 1);
            const uint32_t wv[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              uint32_t h4 = 0, l4 = 0;
#pragma unroll
              for (int f = 0; f < 2; ++f) {
                const uint32_t wd = wv[2 * e + f];
                const float2 a = make_float2(__uint_as_float(wd << 16) * x,
                                             __uint_as_float(wd & 0xffff0000u) * x);
                const __nv_fp8x2_storage_t h = __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E4M3);
                const __half2 hh(__nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3));
                const float2 hf = __half22float2(hh);
                const __nv_fp8x2_storage_t l = __nv_cvt_float2_to_fp8x2(
                    make_float2(a.x - hf.x, a.y - hf.y), __NV_SATFINITE, __NV_E4M3);
                h4 |= (uint32_t)h << (16 * f);
                l4 |= (uint32_t)l << (16 * f);
              }
              hi[e] = h4;
              lo[e] = l4;
            }
            const uint32_t sw = (uint32_t)((k ^ (r & 7)) << 4);  // NH is a multiple of 8
            sts128(qd + r * 128 + sw, hi[0], hi[1], hi[2], hi[3]);
            sts128(qd + (NH + r) * 128 + sw, lo[0], lo[1], lo[2], lo[3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
      }
      if (lane == 0) {
        int* rec = info + kInfoInts * slot;
        rec[kICtx] = w.ctx;
        rec[kIPg0] = w.pg0;
        rec[kIPg1] = w.pg0 + npg;
        rec[kIFlag] = flag;
        rec[kISeq] = w.s;
        rec[kIUnit] = w.unit;
        rec[kIDest] = w.dest;
        rec[kIDone] = item ? 0 : 1;
        rec[kIQInv] = __float_as_int(q_inv);
        if (FP8 || PRO || npg <= 0) {
          mbar_arrive(&B.q_full[slot]);  // FP8, PRO: the rows above are in place
          q_pending[slot] = -1;
        } else if (MULTI) {
          // q as [tokens][Hq][128]: Lg tokens x the G heads of this KV head
          // (rows of a short last group past the sequence's tokens are loaded
          // too and never used)
          const int qh = (w.unit / p.NT) * p.G, qt = w.s * p.L + (w.unit % p.NT) * p.Lg;
          uint8_t* qd = smem + kQ + slot * kOpBytes;
          mbar_arrive_expect_tx(&B.q_full[slot], 2 * p.Lg * p.G * 128);
          tma_load_3d(qd, &tm_q, 0, qh, qt, &B.q_full[slot], pol);
          tma_load_3d(qd + kAtom, &tm_q, 64, qh, qt, &B.q_full[slot], pol);
          q_pending[slot] = (int)((n / kSlots) & 1);
        } else {
          // q as [B * Hq rows][128]: the G consecutive rows of this KV head
          const int qrow = w.s * p.Hq + w.unit * p.G;
          uint8_t* qd = smem + kQ + slot * kOpBytes;
          mbar_arrive_expect_tx(&B.q_full[slot], 2 * p.G * 128);
          tma_load_2d(qd, &tm_q, 0, qrow, &B.q_full[slot], pol);
          tma_load_2d(qd + kAtom, &tm_q, 64, qrow, &B.q_full[slot], pol);
          q_pending[slot] = (int)((n / kSlots) & 1);
        }
      }
      if (!item) break;
      const int x = (w.unit / p.NT) * kHeadDim;
      const int32_t* bt = p.block_table + (int64_t)w.s * p.max_pages;
      for (int c = 0; ok && c < npg; c += 32) {
        const int pid_l = c == 0 ? pid0 : (c + lane < npg ? __ldg(bt + w.pg0 + c + lane) : 0);
        const int cnt = min(32, npg - c);
        for (int k = 0; k < cnt; ++k) {
          const int page = __shfl_sync(0xffffffffu, pid_l, k);
          if (PRO && c + k == npg - 1) {
            // the page holding the new token: its K/V row is stored first
            if (!(ok = mbar_wait_warp(&B.kv_ready[slot], (n / kSlots) & 1, p.status))) break;
          }
          int lok = 1;
          if (lane == 0 && FP8) {
            // e4m3 K and V tiles (128 one-byte dims x 128 tokens each, 128-byte
            // swizzle: the K tile is QK^T's K-major A operand as it lands)
            const int st = gp % kStages8;
            lok = mbar_wait(&B.kv8_empty[st], ((gp / kStages8) & 1) ^ 1, p.status);
            if (lok) {
              uint8_t* dst = smem + kRing8 + st * 2 * kBox8;
              const int y = page * kPage;
              mbar_arrive_expect_tx(&B.k8_full[st], kBox8);
              tma_load_2d(dst, &tm_k, x, y, &B.k8_full[st], pol);
              mbar_arrive_expect_tx(&B.v8_full[st], kBox8);
              tma_load_2d(dst + kBox8, &tm_v, x, y, &B.v8_full[st], pol);
            }
          } else if (lane == 0) {
            const int st = gp % kStages;
            lok = mbar_wait(&B.kv_empty[st], ((gp / kStages) & 1) ^ 1, p.status);
            if (lok) {
              uint8_t* dst = smem + kRing + st * kStageBytes;
              const int y = page * kPage;
              mbar_arrive_expect_tx(&B.k_full[st], 2 * kBox);
              tma_load_2d(dst, &tm_k, x, y, &B.k_full[st], pol);
              tma_load_2d(dst + kBox, &tm_k, x + 64, y, &B.k_full[st], pol);
              mbar_arrive_expect_tx(&B.v_full[st], 2 * kBox);
              tma_load_2d(dst + 2 * kBox, &tm_v, x, y, &B.v_full[st], pol);
              tma_load_2d(dst + 3 * kBox, &tm_v, x + 64, y, &B.v_full[st], pol);
            }
          }
          ok = __shfl_sync(0xffffffffu, lok, 0) != 0;
          if (!ok) break;
          ++gp;
        }
      }
    }
    // drain: copies still in flight (only after a timeout elsewhere) must land
    // before the CTA exits
    if (!tma) {
      // the prologue warp issues no copies
    } else if (lane == 0 && FP8) {
      for (uint32_t g = gp > kStages8 ? gp - kStages8 : 0; g < gp; ++g) {
        mbar_wait(&B.k8_full[g % kStages8], (g / kStages8) & 1, nullptr);
        mbar_wait(&B.v8_full[g % kStages8], (g / kStages8) & 1, nullptr);
      }
    } else if (lane == 0) {
      for (uint32_t g = gp > kStages ? gp - kStages : 0; g < gp; ++g) {
        mbar_wait(&B.k_full[g % kStages], (g / kStages) & 1, nullptr);
        mbar_wait(&B.v_full[g % kStages], (g / kStages) & 1, nullptr);
      }
      for (int k = 0; k < kSlots; ++k)
        if (q_pending[k] >= 0) mbar_wait(&B.q_full[k], (uint32_t)q_pending[k], nullptr);
    }
    __syncwarp();
  } else if (warp == kMmaWarp || (Lay::kSplitIssue && warp == Lay::kPvWarp)) {
    // ------------------------------------------------------------ MMA issuers
    // QK^T of page g goes into S buffer g & 1 and P.V(j) runs once P(j) is
    // in its shared-memory buffer (two, by page parity) and V(j) in the ring;
    // P.V's completion frees the ring stage and the P buffer (K(j) is free
    // too: QK^T(j) finished before the softmax could publish P(j)).
    // One issuing thread (bf16): QK^T(j + 1) before P.V(j), so the tensor
    // core computes the next page's scores while the softmax works on this
    // page's; S buffer g & 1 is free because the thread waited for P(g - 2),
    // and P buffer j & 1 because P.V(j - 2) was issued before QK^T(j).
    // Two (FP8, where one thread's 12 issues per page bound the page period):
    // warp 1 issues QK^T(g) once the softmax has published P(g - 2), warp 14
    // P.V, and the softmax waits for P.V(j - 2) before it writes P(j).
    const bool qk_role = warp == kMmaWarp;
    if (lane == 0) {
      // FP8: e4m3 x e4m3 (format code 0 in kind::f8f6f4), N = the hi and lo columns
      const uint32_t idesc_qk = FP8 ? umma_idesc_e4m3(128, kNS)
                                    : umma_idesc_bf16(128, kN, false, false);
      const uint32_t idesc_pv = FP8 ? umma_idesc_f16(128, kN, true, false)
                                    : umma_idesc_bf16(128, kN, true, false);
      auto qk = [&](uint32_t g, uint32_t q_addr) -> bool {
        if constexpr (Lay::kSplitIssue) {
          if (!mbar_wait(&B.p_full[g & 1], ((g >> 1) & 1) ^ 1, p.status)) return false;
        }
        const uint32_t s_cols = tmem + kColS + (g & 1) * kNS;
        if constexpr (FP8) {
          // A = the e4m3 K tile as TMA landed it (128 keys x 128 bytes,
          // K-major, 128-byte swizzle); 32 dims per instruction
          const int st8 = g % kStages8;
          if (!mbar_wait(&B.k8_full[st8], (g / kStages8) & 1, p.status)) return false;
          tc_fence_after();
          const uint32_t k_addr = smem_u32(smem + kRing8 + st8 * 2 * kBox8);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = umma_sdesc_sw128(k_addr + kk * 32, 16, 1024);
            const uint64_t bd = umma_sdesc_sw128(q_addr + kk * 32, 16, 1024);
            umma_e4m3_ss(s_cols, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
          }
          umma_commit(&B.kv8_empty[st8]);  // the K tile's share of the stage
        } else {
          const int st = g % kStages;
          if (!mbar_wait(&B.k_full[st], (g / kStages) & 1, p.status)) return false;
          tc_fence_after();
          const uint32_t k_addr = smem_u32(smem + kRing + st * kStageBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t ad = umma_sdesc_sw128(k_addr + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = umma_sdesc_sw128(q_addr + (kk >> 2) * kAtom + (kk & 3) * 32, 16, 1024);
            umma_bf16_ss(s_cols, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
          }
        }
        umma_commit(&B.s_full[g & 1]);
        return true;
      };
      auto pv = [&](uint32_t g, bool first, int ob, uint32_t nb) -> bool {
        const int st = g % kStages;
        if (!mbar_wait(&B.p_full[g & 1], (g >> 1) & 1, p.status)) return false;
        if (!mbar_wait(&B.v_full[st], (g / kStages) & 1, p.status)) return false;
        if (first && !mbar_wait(&B.o_free[ob], ((nb >> 1) & 1) ^ 1, p.status)) return false;
        tc_fence_after();
        const uint32_t v_addr = smem_u32(smem + kRing + st * kStageBytes) + (FP8 ? 0 : 2 * kBox);
        const uint32_t p_addr = smem_u32(smem + kP + (g & 1) * kOpBytes);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = umma_sdesc_sw128(v_addr + kk * 2048, kBox, 1024);
          const uint64_t bd = umma_sdesc_sw128(p_addr + (kk >> 2) * kAtom + (kk & 3) * 32, 16, 1024);
          umma_bf16_ss(tmem + kColO + ob * kN, ad, bd, idesc_pv, (!first || kk > 0) ? 1u : 0u);
        }
        umma_commit(&B.kv_empty[st]);
        umma_commit(&B.pv_done[g & 1]);
        return true;
      };
      uint32_t gp = 0, nb = 0;
      bool ok = true;
      for (uint32_t n = 0; ok; ++n) {
        const int slot = n % kSlots;
        if (!(ok = mbar_wait(&B.q_full[slot], (n / kSlots) & 1, p.status))) break;
        const int* rec = info + kInfoInts * slot;
        if (rec[kIDone]) break;
        const int npg = rec[kIPg1] - rec[kIPg0];
        const uint32_t q_addr = smem_u32(smem + kQ + slot * kOpBytes);
        const int ob = nb & 1;
        if (npg <= 0) {
          mbar_arrive(&B.q_empty[slot]);
          continue;
        }
        if (Lay::kSplitIssue && qk_role) {
          for (int j = 0; ok && j < npg; ++j, ++gp) ok = qk(gp, q_addr);
          if (!ok) break;
          umma_commit(&B.q_empty[slot]);  // the query operand is read
          continue;
        }
        if (Lay::kSplitIssue) {
          mbar_arrive(&B.q_empty[slot]);  // the P.V thread reads only the record
          for (int j = 0; ok && j < npg; ++j, ++gp) ok = pv(gp, j == 0, ob, nb);
        } else {
          if (!(ok = qk(gp, q_addr))) break;  // the item's first page
          for (int j = 0; j < npg; ++j, ++gp) {
            // the next page's QK^T runs on the tensor core during this page's softmax
            if (j + 1 < npg && !(ok = qk(gp + 1, q_addr))) break;
            if (j == npg - 1) umma_commit(&B.q_empty[slot]);
            if (!(ok = pv(gp, j == 0, ob, nb))) break;
          }
        }
        if (!ok) break;
        umma_commit(&B.o_full[ob]);
        ++nb;
      }
      // every MMA this thread issued completes before TMEM is released
      umma_commit(B.mma_done);
      mbar_wait(B.mma_done, 0, nullptr);
    }
    __syncwarp();
  } else if (warp >= kConvWarp0) {
    // ------------------------------------------------------------ FP8 V converters, thread = key
    // Each page: wait for its e4m3 V tile and for P.V to be done with the
    // shared-memory stage two pages back, then write V as F16 in the swizzled
    // layout the bf16 path gets from TMA.
    if constexpr (FP8) {
      const int row = (warp & 3) * 32 + lane;  // key 0..127
      const int sw = row & 7;                  // 128-byte swizzle of the row
      uint32_t gp = 0;
      bool ok = true;
      for (uint32_t n = 0; ok; ++n) {
        const int slot = n % kSlots;
        if (!(ok = mbar_wait_warp(&B.q_full[slot], (n / kSlots) & 1, p.status))) break;
        const int* rec = info + kInfoInts * slot;
        if (rec[kIDone]) break;
        const int npg = rec[kIPg1] - rec[kIPg0];
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.q_empty[slot]);
        for (int j = 0; j < npg; ++j, ++gp) {
          const int st8 = gp % kStages8, st = gp % kStages;
          const uint32_t ph = ((gp / kStages) & 1) ^ 1;  // the stage's previous use
          if (!(ok = mbar_wait_warp(&B.v8_full[st8], (gp / kStages8) & 1, p.status))) break;
          if (!(ok = mbar_wait_warp(&B.kv_empty[st], ph, p.status))) break;
          const uint32_t src = smem_u32(smem + kRing8 + st8 * 2 * kBox8 + kBox8) + row * 128;
          const uint32_t dst = smem_u32(smem + kRing + st * kStageBytes) + row * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {  // dims 16c .. 16c + 15
            uint4 lo, hi;
            e4m3x16_to_f16(lds128(src + ((c ^ sw) << 4)), lo, hi);
            const uint32_t d = dst + (c >> 2) * kBox;
            sts128(d + (((2 * (c & 3)) ^ sw) << 4), lo.x, lo.y, lo.z, lo.w);
            sts128(d + (((2 * (c & 3) + 1) ^ sw) << 4), hi.x, hi.y, hi.z, hi.w);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&B.v_full[st]);
            mbar_arrive(&B.kv8_empty[st8]);
          }
        }
      }
    }
  } else if (kN == 32) {
    // ------------------------------------------------------------ 32 columns: softmax + epilogue
    // Warps 2-5 take the item's first 8 or 16 columns, warps 6-9 the rest
    // (at most 16), each group as the 16-column softmax does (thread = key,
    // its own exchange slots), and at the item's end the same threads
    // (thread = head dim) write their columns' outputs.
    const int sg = (warp - kSoftWarp0) >> 2;  // column group
    const int wi = (warp - kSoftWarp0) & 3;
    const int quarter = warp & 3;             // TMEM lanes this warp may access
    const int key = quarter * 32 + lane;      // also the head dim in the epilogue
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    constexpr int kH = 16;                    // columns per group
    float* xbuf = reinterpret_cast<float*>(smem + kX) + sg * 2 * 4 * kH;
    uint64_t* xf = B.x_full + 2 * sg;
    float c = p.scale_log2;
    const int kc = (key & 63) >> 3;
    const uint32_t p_key = (uint32_t)((key >> 6) * kAtom + (key & 7) * 2);
    uint32_t ex = 0;
    auto exchange = [&](const float (&v)[kH], int nv) -> const float* {
      float* slot = xbuf + (ex & 1) * 4 * kH;
      if (lane == 0) {
#pragma unroll
        for (int k = 0; k < kH; ++k)
          if (k < nv) slot[wi * kH + k] = v[k];
        mbar_arrive(&xf[ex & 1]);
      }
      const bool r = mbar_wait_warp(&xf[ex & 1], (ex >> 1) & 1, p.status);
      ++ex;
      return r ? slot : nullptr;
    };
    uint32_t gp = 0, nb = 0;
    bool ok = true;
    for (uint32_t n = 0; ok; ++n) {
      const int slot = n % kSlots;
      if (!(ok = mbar_wait_warp(&B.q_full[slot], (n / kSlots) & 1, p.status))) break;
      const int* rec = info + kInfoInts * slot;
      if (rec[kIDone]) break;
      const int ctx = rec[kICtx], pg0 = rec[kIPg0], pg1 = rec[kIPg1], unit = rec[kIUnit];
      const int flag = rec[kIFlag], sq = rec[kISeq], dest = rec[kIDest];
      const float q_inv = __int_as_float(rec[kIQInv]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.q_empty[slot]);
      const int npg = pg1 - pg0;
      const int GC = MULTI ? unit_columns(p, unit) : p.G;
      // the groups split the item's columns at cb1, a multiple of 8 (so each
      // group's first column is on an 8-column boundary of tensor memory): 8
      // below 24 columns, else 16.  Neither group holds more than 16, and the
      // busier one at most 15 from 17 to 23 columns (a split at 16 would give
      // 20 columns, 4 new tokens of 5 heads, as 16 + 4).
      const int cb1 = GC >= 24 ? 16 : 8;
      const int cb = sg == 0 ? 0 : cb1;  // this group's first column
      const int GL = sg == 0 ? min(GC, cb1) : max(GC - cb1, 0);  // this group's columns
      // FP8: times the item's K scale and 1 / x of its query split
      if constexpr (FP8) c = p.scale_log2 * __ldg(p.k_scale + unit / p.NT) * q_inv;
      // column g = tl * G + head (token t0 + tl) sees key positions below lim[gl]
      int lim[kH];
      {
        int t = (unit % p.NT) * p.Lg + cb / p.G, hg = cb % p.G;
#pragma unroll
        for (int gl = 0; gl < kH; ++gl) {
          lim[gl] = gl < GL ? ctx - (p.L - 1 - t) : 0;
          if (++hg == p.G) {
            hg = 0;
            ++t;
          }
        }
      }
      float res[kH], lse[kH];
      if (npg <= 0) {
        // nothing visible (lse -inf), or an invalid sequence (lse +inf: the
        // combine zeroes the row)
#pragma unroll
        for (int gl = 0; gl < kH; ++gl) {
          res[gl] = 0.f;
          lse[gl] = flag ? INFINITY : -INFINITY;
        }
        if (flag && sg == 0 && wi == 0 && lane == 0 && p.status)
          atomicOr(p.status, flag == 1 ? PA_STATUS_BAD_PAGE : PA_STATUS_BAD_LENGTH);
      } else {
        const int ob = nb & 1;
        float m[kH], ls[kH];
#pragma unroll
        for (int gl = 0; gl < kH; ++gl) {
          m[gl] = -INFINITY;
          ls[gl] = 0.f;
        }
        for (int j = 0; j < npg; ++j, ++gp) {
          const int nvalid = min(ctx - (pg0 + j) * kPage, kPage);  // >= 1
          const bool kv = key < nvalid;
          const int kpos = (pg0 + j) * kPage + key;
          uint32_t vis = 0;
#pragma unroll
          for (int gl = 0; gl < kH; ++gl) vis |= (kpos < lim[gl] ? 1u : 0u) << gl;
          auto visible = [&](int gl) -> bool { return ((vis >> gl) & 1u) != 0; };
          if (!(ok = mbar_wait_warp(&B.s_full[gp & 1], (gp >> 1) & 1, p.status))) break;
          tc_fence_after();
          uint32_t sr[kH];
          const uint32_t s_base = tmem + lane_base + kColS + (gp & 1) * kNS + cb;
          if constexpr (FP8) {
            // scores of the hi and lo query rows (columns NH apart), added
            uint32_t lo[kH];
            tmem_ld8x2(s_base, sr);
            tmem_ld8x2(s_base + NH, lo);
            tmem_wait_ld();
#pragma unroll
            for (int gl = 0; gl < kH; ++gl)
              sr[gl] = __float_as_uint(__uint_as_float(sr[gl]) + __uint_as_float(lo[gl]));
          } else {
            tmem_ld8x2(s_base, sr);
            tmem_wait_ld();
          }
          float d[kH];
          bool need = j == 0;
          if (!need) {
            bool v = false;
#pragma unroll
            for (int gl = 0; gl < kH; ++gl) {
              d[gl] = fmaf(__uint_as_float(sr[gl]), c, -m[gl]);
              if (gl < GL) v |= visible(gl) && d[gl] > kRescaleThreshold;
            }
            float vote[kH];
            vote[0] = __any_sync(0xffffffffu, v) ? 1.f : 0.f;
            const float* x = exchange(vote, 1);
            if (!(ok = x != nullptr)) break;
            need = (x[0] + x[kH]) + (x[2 * kH] + x[3 * kH]) > 0.f;  // uniform over the group
          }
          if (need) {
            float wm[kH];
#pragma unroll
            for (int gl = 0; gl < kH; ++gl)
              wm[gl] = gl < GL ? warp_max(visible(gl) ? __uint_as_float(sr[gl]) * c : -INFINITY) : 0.f;
            const float* x = exchange(wm, GL);
            if (!(ok = x != nullptr)) break;
            float alpha[kH];
#pragma unroll
            for (int gl = 0; gl < kH; ++gl) {
              alpha[gl] = 1.f;
              if (gl < GL) {
                const float M = fmaxf(fmaxf(x[gl], x[kH + gl]), fmaxf(x[2 * kH + gl], x[3 * kH + gl]));
                const float mn = fmaxf(m[gl], M);
                if (j > 0 && mn != -INFINITY) alpha[gl] = fast_exp2(m[gl] - mn);
                m[gl] = mn;
                ls[gl] *= alpha[gl];
              }
              d[gl] = fmaf(__uint_as_float(sr[gl]), c, -m[gl]);
            }
            if (j > 0) {
              if (!(ok = mbar_wait_warp(&B.pv_done[(gp - 1) & 1], ((gp - 1) >> 1) & 1, p.status)))
                break;
              tc_fence_after();
              uint32_t orow[kH];
              const uint32_t o_cols = tmem + lane_base + kColO + ob * kN + cb;
              tmem_ld8x2(o_cols, orow);
              tmem_wait_ld();
#pragma unroll
              for (int gl = 0; gl < kH; ++gl)
                orow[gl] = __float_as_uint(__uint_as_float(orow[gl]) * alpha[gl]);
              tmem_st8x2(o_cols, orow);
            }
          }
          // P(j) into operand buffer j & 1 once P.V(j - 2) has finished reading it
          // (with one issuing thread it has, see the issuers)
          if constexpr (Lay::kSplitIssue) {
            if (!(ok = mbar_wait_warp(&B.pv_done[gp & 1], ((gp >> 1) & 1) ^ 1, p.status))) break;
          }
          const uint32_t pbase = smem_u32(smem + kP + (gp & 1) * kOpBytes) + p_key;
#pragma unroll
          for (int gl = 0; gl < kH; ++gl) {
            if (gl < GL) {
              const int g = cb + gl;
              const float pv = visible(gl) ? fast_exp2(d[gl]) : 0.f;
              uint16_t pbf;
              if constexpr (FP8) {
                const __half ph = __float2half_rn(pv);
                pbf = __half_as_ushort(ph);
                ls[gl] += __half2float(ph);
              } else {
                pbf = __bfloat16_as_ushort(__float2bfloat16_rn(pv));
                ls[gl] += __uint_as_float((uint32_t)pbf << 16);
              }
              sts16(pbase + (g >> 3) * 1024 + (g & 7) * 128 + ((kc ^ (g & 7)) << 4), pbf);
            }
          }
          if (nvalid < kPage && sg == 0) {
            // the sequence's last page: zero the V rows past the context
            const int st = gp % kStages;
            if (!(ok = mbar_wait_warp(&B.v_full[st], (gp / kStages) & 1, p.status))) break;
            if (!kv) {
              const uint32_t vr =
                  smem_u32(smem + kRing + st * kStageBytes + (FP8 ? 0 : 2 * kBox)) + key * 128;
#pragma unroll
              for (int ch = 0; ch < 8; ++ch) {
                sts128(vr + ch * 16, 0u, 0u, 0u, 0u);
                sts128(vr + kBox + ch * 16, 0u, 0u, 0u, 0u);
              }
            }
          }
          fence_proxy_async_smem();
          if (need && j > 0) tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&B.p_full[gp & 1]);
        }
        if (!ok) break;
        // item end: the column sums over the 128 keys, then this group's
        // epilogue once the last P.V is done (thread = head dim)
        float wl[kH];
#pragma unroll
        for (int gl = 0; gl < kH; ++gl) wl[gl] = gl < GL ? warp_sum(ls[gl]) : 0.f;
        const float* x = exchange(wl, GL);
        if (!(ok = x != nullptr)) break;
        const float vsc = FP8 ? __ldg(p.v_scale + unit / p.NT) : 1.f;  // FP8: V scale
        if (!(ok = mbar_wait_warp(&B.o_full[ob], (nb >> 1) & 1, p.status))) break;
        tc_fence_after();
        uint32_t orow[kH];
        tmem_ld8x2(tmem + lane_base + kColO + ob * kN + cb, orow);
        tmem_wait_ld();
#pragma unroll
        for (int gl = 0; gl < kH; ++gl) {
          const float L = (x[gl] + x[kH + gl]) + (x[2 * kH + gl] + x[3 * kH + gl]);
          const float inv = L > 0.f ? vsc / L : 0.f;
          res[gl] = __uint_as_float(orow[gl]) * inv;
          lse[gl] = L > 0.f ? (m[gl] + __log2f(L)) * kLn2 : -INFINITY;
        }
        tc_fence_before();
        mbar_arrive(&B.o_free[ob]);
        ++nb;
      }
      // output row of column g: token t0 + g / G, query head h G + g % G
      const int dim = key;
      const int64_t tok0 = (int64_t)sq * p.L + (unit % p.NT) * p.Lg;
      const int head0 = (unit / p.NT) * p.G;
#pragma unroll
      for (int gl = 0; gl < kH; ++gl) {
        if (gl < GL) {
          const int g = cb + gl;
          const int64_t row = (tok0 + g / p.G) * p.Hq + head0 + g % p.G;
          if (dest < 0) {
            if (p.out_f32)
              reinterpret_cast<float*>(p.out)[row * kHeadDim + dim] = res[gl];
            else
              reinterpret_cast<__nv_bfloat16*>(p.out)[row * kHeadDim + dim] =
                  __float2bfloat16_rn(res[gl]);
          } else if (p.balanced) {
            p.bal_o[((int64_t)dest * kN + g) * kHeadDim + dim] = res[gl];
            if (dim == 0) p.bal_lse[dest * kN + g] = lse[gl];
          } else {
            p.part_o[(row * p.S + dest) * kHeadDim + dim] = res[gl];
            if (dim == 0) p.part_lse[row * p.S + dest] = lse[gl];
          }
        }
      }
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------------------ softmax, thread = key
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int key = quarter * 32 + lane;
    const int wi = warp - kSoftWarp0;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    float* xbuf = reinterpret_cast<float*>(smem + kX);
    float* ml = reinterpret_cast<float*>(smem + kML);
    float c = p.scale_log2;  // FP8: times the item's K scale
    // P^T operand, K-major over keys: row g (head), 64-key atoms, 128-byte swizzle
    const int kc = (key & 63) >> 3;
    const uint32_t p_key = (uint32_t)((key >> 6) * kAtom + (key & 7) * 2);
    // Exchange among the four softmax warps: lane 0 of each warp publishes up
    // to kN floats in slot (ex & 1) and arrives; every warp then waits (bounded)
    // and reads all four rows.  A slot is rewritten two exchanges later, after
    // every warp has arrived at the exchange in between (so has read it).
    uint32_t ex = 0;
    auto exchange = [&](const float (&v)[NH], int nv) -> const float* {
      float* slot = xbuf + (ex & 1) * 4 * kN;
      if (lane == 0) {
#pragma unroll
        for (int k = 0; k < NH; ++k)
          if (k < nv) slot[wi * kN + k] = v[k];
        mbar_arrive(&B.x_full[ex & 1]);
      }
      const bool r = mbar_wait_warp(&B.x_full[ex & 1], (ex >> 1) & 1, p.status);
      ++ex;
      return r ? slot : nullptr;
    };
    uint32_t gp = 0, nb = 0;
    bool ok = true;
    for (uint32_t n = 0; ok; ++n) {
      const int slot = n % kSlots;
      if (!(ok = mbar_wait_warp(&B.q_full[slot], (n / kSlots) & 1, p.status))) break;
      const int* rec = info + kInfoInts * slot;
      if (rec[kIDone]) break;
      const int ctx = rec[kICtx], pg0 = rec[kIPg0], pg1 = rec[kIPg1], unit = rec[kIUnit];
      const float q_inv = __int_as_float(rec[kIQInv]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.q_empty[slot]);
      const int npg = pg1 - pg0;
      if (npg <= 0) continue;
      const int GC = MULTI ? unit_columns(p, unit) : p.G;
      // FP8: times the item's K scale and 1 / x of its query split
      if constexpr (FP8) c = p.scale_log2 * __ldg(p.k_scale + unit / p.NT) * q_inv;
      int lim[NH];
      if constexpr (MULTI) {
        int t = (unit % p.NT) * p.Lg, hg = 0;
#pragma unroll
        for (int g = 0; g < NH; ++g) {
          lim[g] = g < GC ? ctx - (p.L - 1 - t) : 0;
          if (++hg == p.G) {
            hg = 0;
            ++t;
          }
        }
      }
      const int ob = nb & 1;
      float m[NH], ls[NH];
#pragma unroll
      for (int g = 0; g < NH; ++g) {
        m[g] = -INFINITY;
        ls[g] = 0.f;
      }
      for (int j = 0; j < npg; ++j, ++gp) {
        const int nvalid = min(ctx - (pg0 + j) * kPage, kPage);  // >= 1
        const bool kv = key < nvalid;  // within the sequence's context
        const int kpos = (pg0 + j) * kPage + key;
        // MULTI: visible columns of this key, bit g
        uint32_t vis = 0;
        if constexpr (MULTI) {
#pragma unroll
          for (int g = 0; g < NH; ++g) vis |= (kpos < lim[g] ? 1u : 0u) << g;
        }
        auto visible = [&](int g) -> bool { return MULTI ? ((vis >> g) & 1u) != 0 : kv; };
        if (!(ok = mbar_wait_warp(&B.s_full[gp & 1], (gp >> 1) & 1, p.status))) break;
        tc_fence_after();
        uint32_t sr[kN];
        const uint32_t s_base = tmem + lane_base + kColS + (gp & 1) * kNS;
        if constexpr (FP8 && NH == 16) {
          // scores of the hi and lo query rows (columns 16 apart), added
          uint32_t lo[16];
          tmem_ld16(s_base, sr);
          tmem_ld16(s_base + 16, lo);
          tmem_wait_ld();
#pragma unroll
          for (int g = 0; g < 16; ++g)
            sr[g] = __float_as_uint(__uint_as_float(sr[g]) + __uint_as_float(lo[g]));
        } else {
          tmem_ld_cols(s_base, sr);
          tmem_wait_ld();
          if constexpr (FP8) {  // NH == 8: the lo rows' scores are columns 8-15
#pragma unroll
            for (int g = 0; g < 8; ++g)
              sr[g] = __float_as_uint(__uint_as_float(sr[g]) + __uint_as_float(sr[g + 8]));
          }
        }
        float d[NH];
        bool need = j == 0;
        if (!need) {
          bool v = false;
#pragma unroll
          for (int g = 0; g < NH; ++g) {
            d[g] = fmaf(__uint_as_float(sr[g]), c, -m[g]);
            if (g < GC) v |= visible(g) && d[g] > kRescaleThreshold;
          }
          float vote[NH];
          vote[0] = __any_sync(0xffffffffu, v) ? 1.f : 0.f;
          const float* x = exchange(vote, 1);
          if (!(ok = x != nullptr)) break;
          need = (x[0] + x[kN]) + (x[2 * kN] + x[3 * kN]) > 0.f;  // uniform over the 4 warps
        }
        if (need) {
          // exact per-head max of this page; the reference becomes max(m, it)
          float wm[NH];
#pragma unroll
          for (int g = 0; g < NH; ++g)
            wm[g] = g < GC ? warp_max(visible(g) ? __uint_as_float(sr[g]) * c : -INFINITY) : 0.f;
          const float* x = exchange(wm, GC);
          if (!(ok = x != nullptr)) break;
          float alpha[NH];
#pragma unroll
          for (int g = 0; g < NH; ++g) {
            alpha[g] = 1.f;
            if (g < GC) {
              const float M = fmaxf(fmaxf(x[g], x[kN + g]), fmaxf(x[2 * kN + g], x[3 * kN + g]));
              // -inf while the column has seen no visible key (a split that
              // starts past its token's position): nothing to rescale yet
              const float mn = fmaxf(m[g], M);
              if (j > 0 && (!MULTI || mn != -INFINITY)) alpha[g] = fast_exp2(m[g] - mn);
              m[g] = mn;
              ls[g] *= alpha[g];
            }
            d[g] = fmaf(__uint_as_float(sr[g]), c, -m[g]);
          }
          if (j > 0) {
            // O^T holds P.V of the item's earlier pages once the previous
            // page's P.V is done (this page's QK^T was issued before it; the
            // one before it finished ahead of this page's scores)
            if (!(ok = mbar_wait_warp(&B.pv_done[(gp - 1) & 1], ((gp - 1) >> 1) & 1, p.status)))
              break;
            tc_fence_after();
            uint32_t orow[kN];
            const uint32_t o_cols = tmem + lane_base + kColO + ob * kN;
            tmem_ld_cols(o_cols, orow);
            tmem_wait_ld();
#pragma unroll
            for (int g = 0; g < NH; ++g)
              orow[g] = __float_as_uint(__uint_as_float(orow[g]) * alpha[g]);
            tmem_st_cols(o_cols, orow);
          }
        }
        // P(j) into operand buffer j & 1 once P.V(j - 2) has finished reading it
        // (with one issuing thread it has: P.V(j - 2) was issued before QK^T(j),
        // whose commit published these scores)
        if constexpr (Lay::kSplitIssue) {
          if (!(ok = mbar_wait_warp(&B.pv_done[gp & 1], ((gp >> 1) & 1) ^ 1, p.status))) break;
        }
        const uint32_t pbase = smem_u32(smem + kP + (gp & 1) * kOpBytes) + p_key;
#pragma unroll
        for (int g = 0; g < NH; ++g) {
          if (g < GC) {
            const float pv = visible(g) ? fast_exp2(d[g]) : 0.f;
            uint16_t pbf;
            if constexpr (FP8) {
              const __half ph = __float2half_rn(pv);  // the F16 operand
              pbf = __half_as_ushort(ph);
              ls[g] += __half2float(ph);
            } else {
              pbf = __bfloat16_as_ushort(__float2bfloat16_rn(pv));
              ls[g] += __uint_as_float((uint32_t)pbf << 16);
            }
            sts16(pbase + (g >> 3) * 1024 + (g & 7) * 128 + ((kc ^ (g & 7)) << 4), pbf);
          }
        }
        if (nvalid < kPage) {
          // the sequence's last page: zero the V rows past the context
          const int st = gp % kStages;
          if (!(ok = mbar_wait_warp(&B.v_full[st], (gp / kStages) & 1, p.status))) break;
          if (!kv) {
            const uint32_t vr =
                smem_u32(smem + kRing + st * kStageBytes + (FP8 ? 0 : 2 * kBox)) + key * 128;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
              sts128(vr + ch * 16, 0u, 0u, 0u, 0u);
              sts128(vr + kBox + ch * 16, 0u, 0u, 0u, 0u);
            }
          }
        }
        fence_proxy_async_smem();
        if (need && j > 0) tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&B.p_full[gp & 1]);
      }
      if (!ok) break;
      // item end: row sums over the 128 keys, published with the max
      float wl[NH];
#pragma unroll
      for (int g = 0; g < NH; ++g) wl[g] = g < GC ? warp_sum(ls[g]) : 0.f;
      const float* x = exchange(wl, GC);
      if (!(ok = x != nullptr)) break;
      if (wi == 0) {
        if (!(ok = mbar_wait_warp(&B.o_free[ob], ((nb >> 1) & 1) ^ 1, p.status))) break;
        if (lane < GC) {
          float mm = 0.f;
#pragma unroll
          for (int g = 0; g < NH; ++g)
            if (lane == g) mm = m[g];
          ml[(ob * kN + lane) * 2] = mm;
          ml[(ob * kN + lane) * 2 + 1] =
              (x[lane] + x[kN + lane]) + (x[2 * kN + lane] + x[3 * kN + lane]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.ml_full[ob]);
      }
      ++nb;
    }
  } else {
    // ------------------------------------------------------------ epilogue, thread = head dim
    const int quarter = warp & 3;
    const int dim = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const float* ml = reinterpret_cast<const float*>(smem + kML);
    uint32_t nb = 0;
    bool ok = true;
    for (uint32_t n = 0; ok; ++n) {
      const int slot = n % kSlots;
      if (!(ok = mbar_wait_warp(&B.q_full[slot], (n / kSlots) & 1, p.status))) break;
      const int* rec = info + kInfoInts * slot;
      if (rec[kIDone]) break;
      const int pg0 = rec[kIPg0], pg1 = rec[kIPg1], flag = rec[kIFlag];
      const int sq = rec[kISeq], unit = rec[kIUnit], dest = rec[kIDest];
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.q_empty[slot]);
      const int GC = MULTI ? unit_columns(p, unit) : p.G;
      const float vsc = FP8 ? __ldg(p.v_scale + unit / p.NT) : 1.f;  // FP8: V scale
      // output row of column g: token t0 + g / G, query head h G + g % G
      const int64_t tok0 = (int64_t)sq * p.L + (unit % p.NT) * p.Lg;
      const int head0 = (unit / p.NT) * p.G;
      float res[NH], lse[NH];
      if (pg1 - pg0 <= 0) {
        // nothing visible (lse -inf), or an invalid sequence (lse +inf: the
        // combine zeroes the row)
#pragma unroll
        for (int g = 0; g < NH; ++g) {
          res[g] = 0.f;
          lse[g] = flag ? INFINITY : -INFINITY;
        }
        if (flag && warp == kEpiWarp0 && lane == 0 && p.status)
          atomicOr(p.status, flag == 1 ? PA_STATUS_BAD_PAGE : PA_STATUS_BAD_LENGTH);
      } else {
        const int ob = nb & 1;
        if (!(ok = mbar_wait_warp(&B.ml_full[ob], (nb >> 1) & 1, p.status))) break;
        if (!(ok = mbar_wait_warp(&B.o_full[ob], (nb >> 1) & 1, p.status))) break;
        tc_fence_after();
        uint32_t orow[kN];
        tmem_ld_cols(tmem + lane_base + kColO + ob * kN, orow);
        tmem_wait_ld();
#pragma unroll
        for (int g = 0; g < NH; ++g) {
          const float mm = ml[(ob * kN + g) * 2], L = ml[(ob * kN + g) * 2 + 1];
          const float inv = L > 0.f ? vsc / L : 0.f;
          res[g] = __uint_as_float(orow[g]) * inv;
          lse[g] = L > 0.f ? (mm + __log2f(L)) * kLn2 : -INFINITY;
        }
        tc_fence_before();
        mbar_arrive(&B.o_free[ob]);
        ++nb;
      }
      const int64_t row0 = tok0 * p.Hq + head0;
      int64_t row = row0;  // MULTI: column g's row, advanced below
      int hg = 0;
#pragma unroll
      for (int g = 0; g < NH; ++g) {
        if constexpr (MULTI) {
          if (g > 0 && ++hg == p.G) {
            hg = 0;
            row += p.Hq - (p.G - 1);  // next token, first head of the group
          } else if (g > 0) {
            ++row;
          }
        } else {
          row = row0 + g;  // one token: consecutive heads
        }
        if (g < GC) {
          if (dest < 0) {
            if (p.out_f32)
              reinterpret_cast<float*>(p.out)[row * kHeadDim + dim] = res[g];
            else
              reinterpret_cast<__nv_bfloat16*>(p.out)[row * kHeadDim + dim] =
                  __float2bfloat16_rn(res[g]);
          } else if (p.balanced) {
            p.bal_o[((int64_t)dest * kN + g) * kHeadDim + dim] = res[g];
            if (dim == 0) p.bal_lse[dest * kN + g] = lse[g];
          } else {
            p.part_o[(row * p.S + dest) * kHeadDim + dim] = res[g];
            if (dim == 0) p.part_lse[row * p.S + dest] = lse[g];
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::kTmemCols);
  }
}

template <int NH, bool FP8, bool MULTI>
__global__ void __launch_bounds__(Layout<FP8, NH>::kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ DecodeParams p) {
  decode_body<NH, FP8, MULTI, false>(tm_k, tm_v, tm_q, p, nullptr);
}

// The decode step with its prologue (pa_decode_prologue): no q tensor map.
template <int NH>
__global__ void __launch_bounds__(Layout<false, NH>::kThreads + 32, 1)
    decode_prologue_kernel(const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ DecodeParams p,
                           const __grid_constant__ DecodePrologue pro) {
  decode_body<NH, false, false, true>(tm_k, tm_v, tm_k, p, &pro);
}

template <int NH, bool FP8, bool MULTI>
cudaError_t launch_nh(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const CUtensorMap& tm_q,
                      const DecodeParams& p, int num_sms, cudaStream_t stream) {
  constexpr int smem = Layout<FP8, NH>::kSmem, threads = Layout<FP8, NH>::kThreads;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<NH, FP8, MULTI>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = p.balanced ? p.grid : (p.num_items < num_sms ? p.num_items : num_sms);
  if (grid < 1) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode_kernel<NH, FP8, MULTI>, tm_k, tm_v, tm_q, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int NH, bool FP8>
cudaError_t launch_multi(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                         const CUtensorMap& tm_q, const DecodeParams& p, int num_sms,
                         cudaStream_t stream) {
  if constexpr (NH > 16) {
    return launch_nh<NH, FP8, true>(tm_k, tm_v, tm_q, p, num_sms, stream);  // only L > 1 is this wide
  } else {
    return p.L > 1 ? launch_nh<NH, FP8, true>(tm_k, tm_v, tm_q, p, num_sms, stream)
                   : launch_nh<NH, FP8, false>(tm_k, tm_v, tm_q, p, num_sms, stream);
  }
}

template <int NH>
cudaError_t launch_pro_nh(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const DecodeParams& p,
                          const DecodePrologue& pro, int num_sms, cudaStream_t stream) {
  // one more warp than the plain kernel: the prologue warp
  constexpr int smem = Layout<false, NH>::kSmem, threads = Layout<false, NH>::kThreads + 32;
  cudaError_t e = cudaFuncSetAttribute(decode_prologue_kernel<NH>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = p.balanced ? p.grid : (p.num_items < num_sms ? p.num_items : num_sms);
  if (grid < 1) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode_prologue_kernel<NH>, tm_k, tm_v, p, pro);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_prologue(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                   const DecodeParams& p, const DecodePrologue& pro, int g,
                                   int num_sms, cudaStream_t stream) {
  if (g < 1 || g > 16 || p.k_scale || p.L != 1) return cudaErrorInvalidValue;
  return g <= 8 ? launch_pro_nh<8>(tm_k, tm_v, p, pro, num_sms, stream)
                : launch_pro_nh<16>(tm_k, tm_v, p, pro, num_sms, stream);
}

cudaError_t launch_decode(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                          const CUtensorMap& tm_q, const DecodeParams& p, int gc, int num_sms,
                          cudaStream_t stream) {
  if (gc < 1 || gc > 32) return cudaErrorInvalidValue;
  if (p.k_scale)  // FP8 cache
    return gc <= 8    ? launch_multi<8, true>(tm_k, tm_v, tm_q, p, num_sms, stream)
           : gc <= 16 ? launch_multi<16, true>(tm_k, tm_v, tm_q, p, num_sms, stream)
                      : launch_multi<32, true>(tm_k, tm_v, tm_q, p, num_sms, stream);
  return gc <= 8    ? launch_multi<8, false>(tm_k, tm_v, tm_q, p, num_sms, stream)
         : gc <= 16 ? launch_multi<16, false>(tm_k, tm_v, tm_q, p, num_sms, stream)
                    : launch_multi<32, false>(tm_k, tm_v, tm_q, p, num_sms, stream);
}

}  // namespace pa
