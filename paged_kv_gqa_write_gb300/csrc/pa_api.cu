// pa_api.cu -- the extern "C" boundary of libpagedattn.so (declared in
// include/pagedattn.h): host-side argument checks, TMA tensor-map encoding,
// the split-count choice and stream-ordered kernel launches.  Everything the
// path computes runs in the kernels; nothing here touches tensor data.
#include <atomic>
#include <cmath>
#include <mutex>

#include <cudaTypedefs.h>

#include "pa_launch.cuh"

namespace {

using pa::kHeadDim;
using pa::kPage;

constexpr int kMaxGroup = 16;    // query heads per KV head
constexpr int kMaxColumns = 32;  // (token, query head) columns of one decode work item

int check_dims(const pa_dims& d) {
  if (d.head_dim != kHeadDim) return PA_ERR_HEAD_DIM;
  if (d.page_size != kPage) return PA_ERR_PAGE_SIZE;
  if (d.num_kv_heads < 1 || d.num_q_heads < d.num_kv_heads ||
      d.num_q_heads % d.num_kv_heads != 0 || d.num_q_heads / d.num_kv_heads > kMaxGroup)
    return PA_ERR_HEADS;
  if (d.num_seqs < 0 || d.num_pages < 1 || d.max_pages_per_seq < 1) return PA_ERR_DIMS;
  if ((int64_t)d.num_pages * kPage > INT32_MAX) return PA_ERR_DIMS;
  if ((int64_t)d.max_pages_per_seq * kPage > INT32_MAX) return PA_ERR_DIMS;
  if ((int64_t)d.num_kv_heads * kHeadDim > 65536) return PA_ERR_HEADS;
  return PA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Token groups of a decode step with L new tokens per sequence: a work item
// takes Lg tokens x G query heads <= 32 MMA columns.  NT = the fewest groups
// that fit, Lg = the tokens of the largest (groups as even as possible).
void token_groups(int G, int L, int* NT, int* Lg) {
  const int per = kMaxColumns / G;  // >= 1 (G <= 16)
  *NT = (L + per - 1) / per;
  *Lg = (L + *NT - 1) / *NT;
}

int token_group_count(const pa_dims& d, int L) {
  int nt, lg;
  token_groups(d.num_q_heads / d.num_kv_heads, L, &nt, &lg);
  return nt;
}

int device_sms() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (dev >= 0 && dev < 64) {
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (dev >= 0 && dev < 64) cache[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

// Split count for num_splits == 0.  Cost model in units of "page loads on the
// busiest SM", assuming every sequence is full length: rounds of the
// round-robin item deal times (pages per item + a per-item cost of about 2.5
// page loads for the cross-warp merge and pipeline restart), plus about 3.5
// page loads for the combine launch when there is more than one split
// (constants fitted to GB300 sweeps of 16-256 sequences x 4096 tokens).  With
// fewer units than SMs, at least enough splits to give every SM two items.
int auto_splits(const pa_dims& d, int L, int num_sms) {
  const int64_t units = (int64_t)d.num_seqs * d.num_kv_heads * token_group_count(d, L);
  if (units <= 0 || num_sms <= 0) return 1;
  const int mp = d.max_pages_per_seq;
  int best = 1, prev_pps = -1;
  double best_cost = 1e300;
  for (int s = 1; s <= mp; ++s) {
    const int pps = (mp + s - 1) / s;
    if (pps == prev_pps) continue;
    prev_pps = pps;
    const int se = (mp + pps - 1) / pps;
    const int64_t items = units * se;
    const int64_t rounds = (items + num_sms - 1) / num_sms;
    const double cost = rounds * (pps + 2.5) + (se > 1 ? 3.5 : 0.0);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = se;
    }
  }
  if (units < num_sms) {
    const int64_t want = (2 * (int64_t)num_sms + units - 1) / units;
    if (want > best) best = (int)(want < mp ? want : mp);
  }
  return best;
}

// Effective split count and pages per split for a requested count.
void split_shape(const pa_dims& d, int requested, int* splits, int* pps) {
  const int mp = d.max_pages_per_seq;
  int s = requested < 1 ? 1 : (requested > mp ? mp : requested);
  *pps = (mp + s - 1) / s;
  *splits = (mp + *pps - 1) / *pps;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t workspace_bytes_for(const pa_dims& d, int L, int splits) {
  if (splits <= 1) return 0;
  const size_t rows = (size_t)d.num_seqs * L * d.num_q_heads;
  return align256(rows * splits * kHeadDim * sizeof(float)) + align256(rows * splits * sizeof(float));
}

// Partial records of the page-balanced schedule: two per decode CTA, up to
// kMaxColumns column slots of 128 floats plus the lse.
size_t balanced_ws_bytes(int grid) {
  return align256((size_t)2 * grid * kMaxColumns * kHeadDim * sizeof(float)) +
         align256((size_t)2 * grid * kMaxColumns * sizeof(float));
}

// Record columns of the decode kernel for items of gc columns: the MMA width.
int record_columns(int gc) { return gc > 16 ? 32 : 16; }

// Units (KV head x token group) per sequence; the page-balanced schedule runs
// groups of that many CTAs.
int units_per_seq(const pa_dims& d, int L) { return d.num_kv_heads * token_group_count(d, L); }

// The page-balanced schedule takes B <= PA_BALANCED_MAX_SEQS, page positions
// that fit in 31 bits, and at least two CTA groups.
bool balanced_ok(const pa_dims& d, int L, int num_sms) {
  return d.num_seqs <= PA_BALANCED_MAX_SEQS &&
         (int64_t)d.num_seqs * d.max_pages_per_seq < ((int64_t)1 << 31) &&
         num_sms / units_per_seq(d, L) >= 2 && num_sms / units_per_seq(d, L) <= 1024;
}

// The schedule num_splits == 0 selects: 0 for the page-balanced schedule
// (every batch it accepts), else the fixed split count of auto_splits.
int auto_schedule(const pa_dims& d, int L, int num_sms) {
  return balanced_ok(d, L, num_sms) ? 0 : auto_splits(d, L, num_sms);
}

struct DecodePlan {
  bool balanced;
  int splits, pps;  // fixed splits
  int grid;         // page-balanced: CTAs
  size_t ws_bytes;
};

// Resolves num_splits (>= PA_SPLITS_BALANCED) for valid dims with num_seqs > 0;
// false when the request cannot be served.
bool make_plan(const pa_dims& d, int L, int num_splits, int num_sms, DecodePlan* pl) {
  const int req = num_splits == 0 ? auto_schedule(d, L, num_sms) : num_splits;
  if (req == 0 || req == PA_SPLITS_BALANCED) {
    if (!balanced_ok(d, L, num_sms)) return false;
    const int ups = units_per_seq(d, L);
    const int64_t most = (int64_t)d.num_seqs * d.max_pages_per_seq;  // pages at most
    int64_t groups = num_sms / ups;
    if (groups > most) groups = most < 1 ? 1 : most;
    pl->balanced = true;
    pl->splits = 1;
    pl->pps = d.max_pages_per_seq;
    pl->grid = (int)groups * ups;
    pl->ws_bytes = balanced_ws_bytes(pl->grid);
    return true;
  }
  if (req < 1) return false;
  pl->balanced = false;
  split_shape(d, req, &pl->splits, &pl->pps);
  pl->grid = 0;
  pl->ws_bytes = workspace_bytes_for(d, L, pl->splits);
  return true;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 map over a row-major [rows, cols] matrix with the given row pitch
// (bytes), a (box_cols x box_rows) box and the given swizzle.
bool encode_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
               uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows,
               CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D bf16 map over a row-major [d2, d1, d0] array (d0 contiguous) with a
// (box0 x 1 x box2) box: one index of the middle dimension, box2 outer rows.
bool encode_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
               uint32_t box0, uint32_t box2, CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  cuuint32_t box[3] = {box0, 1, box2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// An FP8 (e4m3) cache viewed as [num_pages * 128 rows, Hkv * 128 one-byte
// columns]: 128-byte boxes (one KV head's row) of 128 rows, 128-byte swizzle.
bool encode_cache_map_fp8(CUtensorMap* map, const void* cache, const pa_dims& d) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)d.num_kv_heads * kHeadDim, (cuuint64_t)d.num_pages * kPage};
  cuuint64_t strides[1] = {(cuuint64_t)d.num_kv_heads * kHeadDim};
  cuuint32_t box[2] = {(cuuint32_t)kHeadDim, (cuuint32_t)kPage};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(cache), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The caches viewed as [num_pages * 128 rows, Hkv * 128 columns], row pitch
// Hkv * 128 * 2 bytes; 64-column (128-byte) boxes of 128 rows, 128-byte swizzle.
bool encode_cache_map(CUtensorMap* map, const void* cache, const pa_dims& d) {
  return encode_2d(map, cache, (uint64_t)d.num_kv_heads * kHeadDim,
                   (uint64_t)d.num_pages * kPage, (uint64_t)d.num_kv_heads * kHeadDim * 2, 64,
                   kPage, CU_TENSOR_MAP_SWIZZLE_128B);
}

// q viewed as [B * L tokens][Hq][128]: one item's columns are a box of lg
// tokens x g heads (g x lg rows of 128 elements in shared memory, token-major),
// loaded as two 64-column boxes with 128-byte swizzle.
bool encode_q_decode_map(CUtensorMap* map, const void* q, const pa_dims& d, int L, int g,
                         int lg) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)d.num_q_heads,
                        (cuuint64_t)d.num_seqs * L};
  cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)d.num_q_heads * kHeadDim * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)g, (cuuint32_t)lg};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int launch_result(cudaError_t e) { return e == cudaSuccess ? PA_OK : (int)e; }

// Argument checks shared by pa_decode_multi (and so pa_decode), pa_decode_fp8
// and pa_decode_noalloc, in order: dims, q_len, out_dtype, schedule request;
// then, for a non-empty batch, the row count and the tensor pointers
// (non-null, 16-byte aligned).  *empty is set when there is nothing to launch.
int check_decode_args(const pa_dims& d, int32_t q_len, int32_t out_dtype, int32_t num_splits,
                      const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_table, const int32_t* context_lens, const void* out,
                      bool* empty) {
  *empty = false;
  int rc = check_dims(d);
  if (rc) return rc;
  if (q_len < 1 || q_len > PA_MAX_Q_LEN) return PA_ERR_DIMS;
  if (out_dtype != PA_BF16 && out_dtype != PA_F32) return PA_ERR_OUT_DTYPE;
  if (num_splits < PA_SPLITS_BALANCED) return PA_ERR_SPLITS;
  if (d.num_seqs == 0) {
    *empty = true;
    return PA_OK;
  }
  // rows of q / out are indexed in 32 bits on the device
  if ((int64_t)d.num_seqs * q_len > INT32_MAX / d.num_q_heads) return PA_ERR_DIMS;
  if (!q || !k_cache || !v_cache || !block_table || !context_lens || !out)
    return PA_ERR_NULL_POINTER;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PA_ERR_ALIGNMENT;
  return PA_OK;
}

// Top-k slicing: about two CTAs per SM over all rows, slices of at most 16384
// entries (64 KB of keys in shared memory), a multiple of 4 long.
void topk_plan(int rows, int vocab, int num_sms, int* slices, int* slice_len) {
  const int target = rows > 0 ? (2 * num_sms + rows - 1) / rows : 1;
  int len = (vocab + target - 1) / target;
  if (len < 1024) len = 1024;
  if (len > 16384) len = 16384;
  len = (len + 3) & ~3;
  *slice_len = len;
  *slices = (vocab + len - 1) / len;
}

bool topk_args_ok(int rows, int vocab, int k) {
  return rows >= 0 && k >= 1 && k <= PA_TOPK_MAX_K && vocab >= k && vocab <= (1 << 28);
}

size_t topk_ws_bytes(int rows, int vocab, int k, int num_sms) {
  int slices, len;
  topk_plan(rows, vocab, num_sms, &slices, &len);
  return (size_t)rows * slices * k * sizeof(unsigned long long);
}

// Shared tail of pa_decode, pa_decode_multi and pa_decode_noalloc: arguments
// are checked and `ws` holds at least pl.ws_bytes (or is unused when that is
// 0); q_len new tokens per sequence.
// pro: the step's prologue runs in the decode kernel (q unused).
int run_decode(const void* q, const void* k_cache, const void* v_cache,
               const int32_t* block_table, const int32_t* context_lens, float scale, void* out,
               int32_t out_dtype, uint8_t* ws, const DecodePlan& pl, const pa_dims& d,
               int32_t q_len, int32_t* status, int sms, cudaStream_t st,
               const float* k_scale = nullptr, const float* v_scale = nullptr,
               const pa::DecodePrologue* pro = nullptr) {
  const bool fp8 = k_scale != nullptr;
  const int G = d.num_q_heads / d.num_kv_heads;
  int NT, Lg;
  token_groups(G, q_len, &NT, &Lg);
  const int64_t items = (int64_t)pl.splits * d.num_seqs * d.num_kv_heads * NT;
  if (items > INT32_MAX) return PA_ERR_DIMS;
  CUtensorMap tm_k, tm_v, tm_q;
  const bool maps_ok = fp8 ? encode_cache_map_fp8(&tm_k, k_cache, d) &&
                                 encode_cache_map_fp8(&tm_v, v_cache, d)
                           : encode_cache_map(&tm_k, k_cache, d) &&
                                 encode_cache_map(&tm_v, v_cache, d);
  // one token per sequence: q as [B * Hq rows, 128] with G-row boxes; more: a
  // 3-D map over [tokens][Hq][128] with (G heads x Lg tokens) boxes
  const bool q_ok = pro ? true
                 : q_len == 1 ? encode_2d(&tm_q, q, kHeadDim, (uint64_t)d.num_seqs * d.num_q_heads,
                                          kHeadDim * 2, 64, (uint32_t)G, CU_TENSOR_MAP_SWIZZLE_128B)
                              : encode_q_decode_map(&tm_q, q, d, q_len, G, Lg);
  if (!maps_ok || !q_ok) return PA_ERR_TENSOR_MAP;

  pa::DecodeParams p = {};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.block_table = block_table;
  p.context_lens = context_lens;
  p.out = out;
  const size_t rows = (size_t)d.num_seqs * q_len * d.num_q_heads;
  const bool fixed_parts = !pl.balanced && pl.splits > 1;
  p.part_o = fixed_parts ? reinterpret_cast<float*>(ws) : nullptr;
  p.part_lse = fixed_parts ? reinterpret_cast<float*>(ws + align256(rows * pl.splits * kHeadDim * 4))
                           : nullptr;
  p.status = status;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.B = d.num_seqs;
  p.Hq = d.num_q_heads;
  p.Hkv = d.num_kv_heads;
  p.G = G;
  p.L = q_len;
  p.NT = NT;
  p.Lg = Lg;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.num_pages = d.num_pages;
  p.max_pages = d.max_pages_per_seq;
  p.pps = pl.pps;
  p.S = pl.splits;
  p.num_items = (int32_t)items;
  p.out_f32 = out_dtype == PA_F32;
  p.balanced = pl.balanced ? 1 : 0;
  p.grid = pl.grid;
  p.bal_o = pl.balanced ? reinterpret_cast<float*>(ws) : nullptr;
  p.bal_lse = pl.balanced ? reinterpret_cast<float*>(
                                ws + align256((size_t)2 * pl.grid * kMaxColumns * kHeadDim *
                                              sizeof(float)))
                          : nullptr;
  cudaError_t e = pro ? pa::launch_decode_prologue(tm_k, tm_v, p, *pro, G, sms, st)
                      : pa::launch_decode(tm_k, tm_v, tm_q, p, G * Lg, sms, st);
  if (e != cudaSuccess) return launch_result(e);
  if (pl.balanced) {
    pa::BalCombineParams c;
    c.context_lens = context_lens;
    c.bal_o = p.bal_o;
    c.bal_lse = p.bal_lse;
    c.out = out;
    c.B = d.num_seqs;
    c.Hq = d.num_q_heads;
    c.G = G;
    c.max_pages = d.max_pages_per_seq;
    c.L = q_len;
    c.NT = NT;
    c.Lg = Lg;
    c.grid = pl.grid;
    c.NC = record_columns(G * Lg);
    c.out_f32 = p.out_f32;
    return launch_result(pa::launch_bal_combine(c, st));
  }
  if (pl.splits == 1) return PA_OK;
  pa::CombineParams c;
  c.part_o = p.part_o;
  c.part_lse = p.part_lse;
  c.out = out;
  c.rows = (int32_t)rows;
  c.S = pl.splits;
  c.out_f32 = p.out_f32;
  return launch_result(pa::launch_combine(c, st));
}

}  // namespace

extern "C" {

int32_t pa_abi_version(void) { return 106; }

const char* pa_status_string(int32_t code) {
  switch (code) {
    case PA_OK: return "ok";
    case PA_ERR_NULL_POINTER: return "a required pointer is NULL";
    case PA_ERR_HEAD_DIM: return "head_dim must be 128";
    case PA_ERR_PAGE_SIZE: return "page_size must be 128";
    case PA_ERR_HEADS: return "num_q_heads must be a multiple of num_kv_heads with ratio <= 16";
    case PA_ERR_DIMS: return "invalid num_seqs / num_pages / max_pages_per_seq / num_tokens";
    case PA_ERR_ALIGNMENT: return "a tensor pointer is not 16-byte aligned";
    case PA_ERR_OUT_DTYPE: return "out_dtype must be PA_BF16 or PA_F32";
    case PA_ERR_WORKSPACE: return "workspace is NULL or smaller than pa_decode_workspace_size()";
    case PA_ERR_SPLITS:
      return "num_splits must be >= 0, or PA_SPLITS_BALANCED with num_seqs <= PA_BALANCED_MAX_SEQS";
    case PA_ERR_TOO_MANY_SEQS: return "num_seqs exceeds PA_MAX_CHUNKED_SEQS for a chunked call";
    case PA_ERR_TENSOR_MAP: return "TMA tensor map encoding failed";
    case PA_ERR_NO_DEVICE: return "no CUDA device is current";
    case PA_ERR_NOALLOC_TOO_LARGE:
      return "split partials exceed PA_NOALLOC_SCRATCH_BYTES: use fewer splits or pa_decode";
    default: break;
  }
  if (code > 0) return cudaGetErrorString(static_cast<cudaError_t>(code));
  return "unknown status";
}

}  // extern "C"

namespace {

int kv_write_impl(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                  const float* k_scale, const float* v_scale, const int32_t* block_table,
                  const int32_t* context_lens, const int32_t* chunk_lens, int32_t num_tokens,
                  pa_dims d, int32_t* status, pa_stream_t stream) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (num_tokens < 0) return PA_ERR_DIMS;
  if (!chunk_lens && num_tokens != d.num_seqs) return PA_ERR_DIMS;
  if (chunk_lens && d.num_seqs > PA_MAX_CHUNKED_SEQS) return PA_ERR_TOO_MANY_SEQS;
  if (num_tokens == 0 || d.num_seqs == 0) return PA_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !context_lens)
    return PA_ERR_NULL_POINTER;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_ALIGNMENT;
  const int sms = device_sms();
  if (sms <= 0) return PA_ERR_NO_DEVICE;
  pa::KvWriteParams p;
  p.k_new = static_cast<const uint4*>(k_new);
  p.v_new = static_cast<const uint4*>(v_new);
  p.k_cache = static_cast<uint4*>(k_cache);
  p.v_cache = static_cast<uint4*>(v_cache);
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.block_table = block_table;
  p.context_lens = context_lens;
  p.chunk_lens = chunk_lens;
  p.status = status;
  p.B = d.num_seqs;
  p.T = num_tokens;
  p.Hkv = d.num_kv_heads;
  p.num_pages = d.num_pages;
  p.max_pages = d.max_pages_per_seq;
  return launch_result(pa::launch_kv_write(p, sms, reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

int pa_kv_write(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                const int32_t* block_table, const int32_t* context_lens,
                const int32_t* chunk_lens, int32_t num_tokens, pa_dims d, int32_t* status,
                pa_stream_t stream) {
  return kv_write_impl(k_new, v_new, k_cache, v_cache, nullptr, nullptr, block_table,
                       context_lens, chunk_lens, num_tokens, d, status, stream);
}

int pa_kv_write_fp8(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                    const float* k_scale, const float* v_scale, const int32_t* block_table,
                    const int32_t* context_lens, const int32_t* chunk_lens, int32_t num_tokens,
                    pa_dims d, int32_t* status, pa_stream_t stream) {
  if (!k_scale || !v_scale) return PA_ERR_NULL_POINTER;
  if (((reinterpret_cast<uintptr_t>(k_scale) | reinterpret_cast<uintptr_t>(v_scale)) & 3u) != 0)
    return PA_ERR_ALIGNMENT;
  return kv_write_impl(k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_table,
                       context_lens, chunk_lens, num_tokens, d, status, stream);
}

namespace {

// The 64 NeoX pairs' frequencies base^(-2i/D) / scale in radians per position
// (double) and in turns per position as an unevaluated float pair hi + lo.
void rope_tables(float rope_base, float rope_scale, double* freq, float* turn_hi,
                 float* turn_lo) {
  const double log2_base = std::log2((double)rope_base);
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < 64; ++i) {
    const double f = std::exp2(-2.0 * i / kHeadDim * log2_base) / (double)rope_scale;
    const double g = f / two_pi;
    freq[i] = f;
    turn_hi[i] = (float)g;
    turn_lo[i] = (float)(g - (double)turn_hi[i]);
  }
}

bool prologue_scalars_ok(float eps, float rope_base, float rope_scale, float q_scale) {
  return eps >= 0.f && rope_base > 0.f && rope_scale > 0.f && std::isfinite(eps) &&
         std::isfinite(rope_base) && std::isfinite(rope_scale) && std::isfinite(q_scale);
}

// The prologue into a bf16 cache (k_scale == v_scale == null) or an FP8 one.
int prologue_impl(const void* qkv, const float* q_norm_w, const float* k_norm_w, float eps,
                  float rope_base, float rope_scale, float q_scale, void* q_out, void* k_cache,
                  void* v_cache, const float* k_scale, const float* v_scale,
                  const int32_t* block_table, const int32_t* context_lens,
                  const int32_t* chunk_lens, int32_t num_tokens, pa_dims d, int32_t* status,
                  pa_stream_t stream) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (num_tokens < 0) return PA_ERR_DIMS;
  if (!chunk_lens && num_tokens != d.num_seqs) return PA_ERR_DIMS;
  if (chunk_lens && d.num_seqs > PA_MAX_CHUNKED_SEQS) return PA_ERR_TOO_MANY_SEQS;
  if (d.num_q_heads + 2 * d.num_kv_heads > PA_MAX_PROLOGUE_HEADS) return PA_ERR_HEADS;
  if (!prologue_scalars_ok(eps, rope_base, rope_scale, q_scale)) return PA_ERR_DIMS;
  if (num_tokens == 0 || d.num_seqs == 0) return PA_OK;
  if (!qkv || !q_norm_w || !k_norm_w || !q_out || !k_cache || !v_cache || !block_table ||
      !context_lens)
    return PA_ERR_NULL_POINTER;
  if (!aligned16(qkv) || !aligned16(q_norm_w) || !aligned16(k_norm_w) || !aligned16(q_out) ||
      !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_ALIGNMENT;
  const int sms = device_sms();
  if (sms <= 0) return PA_ERR_NO_DEVICE;
  pa::PrologueParams p;
  p.qkv = static_cast<const uint2*>(qkv);
  p.wq = q_norm_w;
  p.wk = k_norm_w;
  p.q_out = static_cast<uint2*>(q_out);
  p.k_cache = static_cast<uint2*>(k_cache);
  p.v_cache = static_cast<uint2*>(v_cache);
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.block_table = block_table;
  p.context_lens = context_lens;
  p.chunk_lens = chunk_lens;
  p.status = status;
  p.eps = eps;
  p.q_scale = q_scale;
  rope_tables(rope_base, rope_scale, p.freq, p.turn_hi, p.turn_lo);
  p.B = d.num_seqs;
  p.T = num_tokens;
  p.Hq = d.num_q_heads;
  p.Hkv = d.num_kv_heads;
  p.num_pages = d.num_pages;
  p.max_pages = d.max_pages_per_seq;
  return launch_result(pa::launch_prologue(p, sms, reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

int pa_qk_norm_rope_write(const void* qkv, const float* q_norm_w, const float* k_norm_w,
                          float eps, float rope_base, float rope_scale, float q_scale,
                          void* q_out, void* k_cache, void* v_cache,
                          const int32_t* block_table, const int32_t* context_lens,
                          const int32_t* chunk_lens, int32_t num_tokens, pa_dims d,
                          int32_t* status, pa_stream_t stream) {
  return prologue_impl(qkv, q_norm_w, k_norm_w, eps, rope_base, rope_scale, q_scale, q_out,
                       k_cache, v_cache, nullptr, nullptr, block_table, context_lens,
                       chunk_lens, num_tokens, d, status, stream);
}

int pa_qk_norm_rope_write_fp8(const void* qkv, const float* q_norm_w, const float* k_norm_w,
                              float eps, float rope_base, float rope_scale, float q_scale,
                              void* q_out, void* k_cache, void* v_cache, const float* k_scale,
                              const float* v_scale, const int32_t* block_table,
                              const int32_t* context_lens, const int32_t* chunk_lens,
                              int32_t num_tokens, pa_dims d, int32_t* status,
                              pa_stream_t stream) {
  if (!k_scale || !v_scale) return PA_ERR_NULL_POINTER;
  if (((reinterpret_cast<uintptr_t>(k_scale) | reinterpret_cast<uintptr_t>(v_scale)) & 3u) != 0)
    return PA_ERR_ALIGNMENT;
  return prologue_impl(qkv, q_norm_w, k_norm_w, eps, rope_base, rope_scale, q_scale, q_out,
                       k_cache, v_cache, k_scale, v_scale, block_table, context_lens,
                       chunk_lens, num_tokens, d, status, stream);
}

size_t pa_topk_workspace_size(int32_t rows, int32_t vocab, int32_t k) {
  if (!topk_args_ok(rows, vocab, k)) return (size_t)-1;
  const int sms = device_sms();
  if (sms <= 0) return (size_t)-1;
  return topk_ws_bytes(rows, vocab, k, sms);
}

int pa_topk(const float* logits, int64_t row_stride, int32_t rows, int32_t vocab, int32_t k,
            float* out_values, int32_t* out_indices, void* workspace, size_t ws_bytes,
            pa_stream_t stream) {
  if (!topk_args_ok(rows, vocab, k) || row_stride < vocab) return PA_ERR_DIMS;
  if (rows == 0) return PA_OK;
  if (!logits || !out_values || !out_indices || !workspace) return PA_ERR_NULL_POINTER;
  if ((reinterpret_cast<uintptr_t>(logits) & 3u) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(out_values) & 3u) || (reinterpret_cast<uintptr_t>(out_indices) & 3u))
    return PA_ERR_ALIGNMENT;
  const int sms = device_sms();
  if (sms <= 0) return PA_ERR_NO_DEVICE;
  if (ws_bytes < topk_ws_bytes(rows, vocab, k, sms)) return PA_ERR_WORKSPACE;
  pa::TopkParams p;
  p.logits = logits;
  p.row_stride = row_stride;
  p.out_values = out_values;
  p.out_indices = out_indices;
  p.cand = static_cast<unsigned long long*>(workspace);
  p.rows = rows;
  p.vocab = vocab;
  p.k = k;
  topk_plan(rows, vocab, sms, &p.slices, &p.slice_len);
  if ((int64_t)p.slices * k * 8 > 200 * 1024) return PA_ERR_DIMS;
  return launch_result(pa::launch_topk(p, reinterpret_cast<cudaStream_t>(stream)));
}

int32_t pa_decode_auto_splits(pa_dims d) {
  int rc = check_dims(d);
  if (rc) return rc;
  const int sms = device_sms();
  if (sms <= 0) return PA_ERR_NO_DEVICE;
  return auto_schedule(d, 1, sms);
}

size_t pa_decode_multi_workspace_size(pa_dims d, int32_t q_len, int32_t num_splits) {
  if (check_dims(d) || num_splits < PA_SPLITS_BALANCED) return (size_t)-1;
  if (q_len < 1 || q_len > PA_MAX_Q_LEN) return (size_t)-1;
  if (d.num_seqs == 0) return 0;
  if ((int64_t)d.num_seqs * q_len > INT32_MAX / d.num_q_heads) return (size_t)-1;
  const int sms = device_sms();
  if (sms <= 0) return (size_t)-1;
  DecodePlan pl;
  if (!make_plan(d, q_len, num_splits, sms, &pl)) return (size_t)-1;
  return pl.ws_bytes;
}

size_t pa_decode_workspace_size(pa_dims d, int32_t num_splits) {
  return pa_decode_multi_workspace_size(d, 1, num_splits);
}

int pa_decode_multi(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_table, const int32_t* context_lens, int32_t q_len,
                    float scale, void* out, int32_t out_dtype, void* workspace, size_t ws_bytes,
                    int32_t num_splits, pa_dims d, int32_t* status, pa_stream_t stream) {
  bool empty = false;
  int rc = check_decode_args(d, q_len, out_dtype, num_splits, q, k_cache, v_cache, block_table,
                             context_lens, out, &empty);
  if (rc || empty) return rc;
  const int sms = device_sms();
  if (sms <= 0) return PA_ERR_NO_DEVICE;
  DecodePlan pl;
  if (!make_plan(d, q_len, num_splits, sms, &pl)) return PA_ERR_SPLITS;
  if (pl.ws_bytes > 0) {
    if (!workspace || ws_bytes < pl.ws_bytes) return PA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PA_ERR_ALIGNMENT;
  }
  return run_decode(q, k_cache, v_cache, block_table, context_lens, scale, out, out_dtype,
                    static_cast<uint8_t*>(workspace), pl, d, q_len, status, sms,
                    reinterpret_cast<cudaStream_t>(stream));
}

int pa_decode(const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_table, const int32_t* context_lens, float scale, void* out,
              int32_t out_dtype, void* workspace, size_t ws_bytes, int32_t num_splits,
              pa_dims d, int32_t* status, pa_stream_t stream) {
  return pa_decode_multi(q, k_cache, v_cache, block_table, context_lens, 1, scale, out,
                         out_dtype, workspace, ws_bytes, num_splits, d, status, stream);
}

int pa_decode_prologue(const void* qkv, const float* q_norm_w, const float* k_norm_w, float eps,
                       float rope_base, float rope_scale, float q_scale, void* k_cache,
                       void* v_cache, const int32_t* block_table, const int32_t* context_lens,
                       float scale, void* out, int32_t out_dtype, void* workspace,
                       size_t ws_bytes, int32_t num_splits, pa_dims d, int32_t* status,
                       pa_stream_t stream) {
  bool empty = false;
  int rc = check_decode_args(d, 1, out_dtype, num_splits, qkv, k_cache, v_cache, block_table,
                             context_lens, out, &empty);
  if (rc) return rc;
  if (d.num_q_heads / d.num_kv_heads > 16) return PA_ERR_HEADS;
  if (!prologue_scalars_ok(eps, rope_base, rope_scale, q_scale)) return PA_ERR_DIMS;
  if (empty) return PA_OK;
  if (!q_norm_w || !k_norm_w) return PA_ERR_NULL_POINTER;
  if (!aligned16(q_norm_w) || !aligned16(k_norm_w)) return PA_ERR_ALIGNMENT;
  const int sms = device_sms();
  if (sms <= 0) return PA_ERR_NO_DEVICE;
  DecodePlan pl;
  if (!make_plan(d, 1, num_splits, sms, &pl)) return PA_ERR_SPLITS;
  if (pl.ws_bytes > 0) {
    if (!workspace || ws_bytes < pl.ws_bytes) return PA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PA_ERR_ALIGNMENT;
  }
  pa::DecodePrologue pro = {};
  pro.qkv = static_cast<const __nv_bfloat16*>(qkv);
  pro.wq = q_norm_w;
  pro.wk = k_norm_w;
  pro.k_cache = static_cast<__nv_bfloat16*>(k_cache);
  pro.v_cache = static_cast<__nv_bfloat16*>(v_cache);
  pro.eps = eps;
  pro.q_scale = q_scale;
  rope_tables(rope_base, rope_scale, pro.freq, pro.turn_hi, pro.turn_lo);
  return run_decode(nullptr, k_cache, v_cache, block_table, context_lens, scale, out, out_dtype,
                    static_cast<uint8_t*>(workspace), pl, d, 1, status, sms,
                    reinterpret_cast<cudaStream_t>(stream), nullptr, nullptr, &pro);
}

int pa_decode_fp8(const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                  const float* v_scale, const int32_t* block_table,
                  const int32_t* context_lens, int32_t q_len, float scale, void* out,
                  int32_t out_dtype, void* workspace, size_t ws_bytes, int32_t num_splits,
                  pa_dims d, int32_t* status, pa_stream_t stream) {
  bool empty = false;
  int rc = check_decode_args(d, q_len, out_dtype, num_splits, q, k_cache, v_cache, block_table,
                             context_lens, out, &empty);
  if (rc || empty) return rc;
  if (!k_scale || !v_scale) return PA_ERR_NULL_POINTER;
  if (((reinterpret_cast<uintptr_t>(k_scale) | reinterpret_cast<uintptr_t>(v_scale)) & 3u) != 0)
    return PA_ERR_ALIGNMENT;
  const int sms = device_sms();
  if (sms <= 0) return PA_ERR_NO_DEVICE;
  DecodePlan pl;
  if (!make_plan(d, q_len, num_splits, sms, &pl)) return PA_ERR_SPLITS;
  if (pl.ws_bytes > 0) {
    if (!workspace || ws_bytes < pl.ws_bytes) return PA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PA_ERR_ALIGNMENT;
  }
  return run_decode(q, k_cache, v_cache, block_table, context_lens, scale, out, out_dtype,
                    static_cast<uint8_t*>(workspace), pl, d, q_len, status, sms,
                    reinterpret_cast<cudaStream_t>(stream), k_scale, v_scale);
}

int pa_combine(const float* part_o, const float* part_lse, int32_t num_splits, void* out,
               int32_t out_dtype, pa_dims d, pa_stream_t stream) {
  if (d.head_dim != kHeadDim) return PA_ERR_HEAD_DIM;
  if (d.num_seqs < 0 || d.num_q_heads < 1) return PA_ERR_DIMS;
  if (num_splits < 1) return PA_ERR_SPLITS;
  if (out_dtype != PA_BF16 && out_dtype != PA_F32) return PA_ERR_OUT_DTYPE;
  const int64_t rows = (int64_t)d.num_seqs * d.num_q_heads;
  if (rows == 0) return PA_OK;
  if (rows > INT32_MAX) return PA_ERR_DIMS;
  if (!part_o || !part_lse || !out) return PA_ERR_NULL_POINTER;
  if (!aligned16(part_o) || !aligned16(out) || (reinterpret_cast<uintptr_t>(part_lse) & 3u))
    return PA_ERR_ALIGNMENT;
  pa::CombineParams c;
  c.part_o = part_o;
  c.part_lse = part_lse;
  c.out = out;
  c.rows = (int32_t)rows;
  c.S = num_splits;
  c.out_f32 = out_dtype == PA_F32;
  return launch_result(pa::launch_combine(c, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// An FP8 (e4m3) cache viewed as [num_pages * 128 rows, Hkv * 128 one-byte
// columns] with the given box and swizzle.
bool encode_cache_u8(CUtensorMap* map, const void* cache, const pa_dims& d, uint32_t box_cols,
                     uint32_t box_rows, CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)d.num_kv_heads * kHeadDim, (cuuint64_t)d.num_pages * kPage};
  cuuint64_t strides[1] = {(cuuint64_t)d.num_kv_heads * kHeadDim};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(cache), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// pa_prefill_chunk over a bf16 cache (k_scale == nullptr) or an FP8 one.
int prefill_impl(const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                 const float* v_scale, const int32_t* block_table, const int32_t* context_lens,
                 const int32_t* chunk_lens, int32_t num_tokens, float scale, void* out,
                 int32_t out_dtype, pa_dims d, int32_t* status, pa_stream_t stream) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (out_dtype != PA_BF16 && out_dtype != PA_F32) return PA_ERR_OUT_DTYPE;
  if (num_tokens < 0) return PA_ERR_DIMS;
  if (d.num_seqs > PA_MAX_CHUNKED_SEQS) return PA_ERR_TOO_MANY_SEQS;
  if (num_tokens == 0 || d.num_seqs == 0) return PA_OK;
  if (!q || !k_cache || !v_cache || !block_table || !context_lens || !chunk_lens || !out)
    return PA_ERR_NULL_POINTER;
  const bool fp8 = k_scale != nullptr;
  if (fp8 && !v_scale) return PA_ERR_NULL_POINTER;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PA_ERR_ALIGNMENT;
  if (fp8 && ((reinterpret_cast<uintptr_t>(k_scale) | reinterpret_cast<uintptr_t>(v_scale)) & 3u))
    return PA_ERR_ALIGNMENT;
  if ((int64_t)num_tokens * d.num_q_heads * kHeadDim > ((int64_t)1 << 40)) return PA_ERR_DIMS;
  const int sms = device_sms();
  if (sms <= 0) return PA_ERR_NO_DEVICE;
  CUtensorMap tm_k, tm_v, tm_q;
  // each CTA of a pair stages half a page tile: K as 64-key boxes (64 dims
  // wide, or all 128 one-byte dims of an e4m3 row), V as 128-key x 64-dim
  // boxes
  const bool maps_ok =
      fp8 ? encode_cache_u8(&tm_k, k_cache, d, kHeadDim, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
                encode_cache_u8(&tm_v, v_cache, d, 64, kPage, CU_TENSOR_MAP_SWIZZLE_64B)
          : encode_2d(&tm_k, k_cache, (uint64_t)d.num_kv_heads * kHeadDim,
                      (uint64_t)d.num_pages * kPage, (uint64_t)d.num_kv_heads * kHeadDim * 2, 64,
                      64, CU_TENSOR_MAP_SWIZZLE_128B) &&
                encode_cache_map(&tm_v, v_cache, d);
  if (!maps_ok) return PA_ERR_TENSOR_MAP;
  // q as [num_tokens, Hq, 128]: a box is 128 tokens of one head, 64 dims wide.
  if (!encode_3d(&tm_q, q, kHeadDim, d.num_q_heads, (uint64_t)num_tokens, 64, 128,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return PA_ERR_TENSOR_MAP;
  // out as [num_tokens, Hq, 128] for the BF16 output tiles' TMA stores
  CUtensorMap tm_o = {};
  if (out_dtype == PA_BF16 &&
      !encode_3d(&tm_o, out, kHeadDim, d.num_q_heads, (uint64_t)num_tokens, 64, 128,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return PA_ERR_TENSOR_MAP;
  pa::PrefillParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.block_table = block_table;
  p.context_lens = context_lens;
  p.chunk_lens = chunk_lens;
  p.out = out;
  p.status = status;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.B = d.num_seqs;
  p.T = num_tokens;
  p.Hq = d.num_q_heads;
  p.Hkv = d.num_kv_heads;
  p.G = d.num_q_heads / d.num_kv_heads;
  p.num_pages = d.num_pages;
  p.max_pages = d.max_pages_per_seq;
  p.out_f32 = out_dtype == PA_F32;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  return launch_result(
      pa::launch_prefill(tm_k, tm_v, tm_q, tm_o, p, sms, reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

int pa_prefill_chunk(const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_table, const int32_t* context_lens,
                     const int32_t* chunk_lens, int32_t num_tokens, float scale, void* out,
                     int32_t out_dtype, pa_dims d, int32_t* status, pa_stream_t stream) {
  return prefill_impl(q, k_cache, v_cache, nullptr, nullptr, block_table, context_lens,
                      chunk_lens, num_tokens, scale, out, out_dtype, d, status, stream);
}

int pa_prefill_chunk_fp8(const void* q, const void* k_cache, const void* v_cache,
                         const float* k_scale, const float* v_scale, const int32_t* block_table,
                         const int32_t* context_lens, const int32_t* chunk_lens,
                         int32_t num_tokens, float scale, void* out, int32_t out_dtype,
                         pa_dims d, int32_t* status, pa_stream_t stream) {
  if (!k_scale || !v_scale) return PA_ERR_NULL_POINTER;
  return prefill_impl(q, k_cache, v_cache, k_scale, v_scale, block_table, context_lens,
                      chunk_lens, num_tokens, scale, out, out_dtype, d, status, stream);
}

int32_t pa_prefill_pairs(void) {
  const int sms = device_sms();
  if (sms <= 0) return PA_ERR_NO_DEVICE;
  int pairs = 0;
  const cudaError_t e = pa::prefill_pairs(sms, &pairs);
  return e == cudaSuccess ? pairs : launch_result(e);
}

int pa_wait_selftest(uint32_t limit_us, int32_t* status, pa_stream_t stream) {
  if (limit_us < 1 || limit_us > 5000000u) return PA_ERR_DIMS;
  if (!status) return PA_ERR_NULL_POINTER;
  return launch_result(pa::launch_wait_selftest((uint64_t)limit_us * 1000u, status,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// pa_decode_noalloc: pa_decode for callers that cannot allocate device memory.
//
// The split partials live in one file-scope device array instead of a
// caller-provided workspace.  Its device address is looked up once per device
// (on the first call made with that device current) and cached; host code
// must never hand the symbol itself to a kernel, because on the host the name
// refers to a host-side stand-in, not to device memory.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

// Device address of g_noalloc_scratch on the current device, or null with
// *err set when the lookup fails.
void* noalloc_scratch(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    *err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    g_noalloc_ptr[dev] = ptr;
  }
  return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" int pa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_table, const int32_t* context_lens,
                                 float scale, void* out, int32_t out_dtype, int32_t num_splits,
                                 pa_dims d, int32_t* status, pa_stream_t stream) {
  bool empty = false;
  int rc = check_decode_args(d, 1, out_dtype, num_splits, q, k_cache, v_cache, block_table,
                             context_lens, out, &empty);
  if (rc || empty) return rc;
  const int sms = device_sms();
  if (sms <= 0) return PA_ERR_NO_DEVICE;
  DecodePlan pl;
  if (!make_plan(d, 1, num_splits, sms, &pl)) return PA_ERR_SPLITS;
  if (pl.ws_bytes > PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_NOALLOC_TOO_LARGE;
  uint8_t* scratch = nullptr;
  if (pl.ws_bytes > 0) {
    cudaError_t e = cudaSuccess;
    scratch = static_cast<uint8_t*>(noalloc_scratch(&e));
    if (!scratch) return launch_result(e == cudaSuccess ? cudaErrorUnknown : e);
  }
  return run_decode(q, k_cache, v_cache, block_table, context_lens, scale, out, out_dtype,
                    scratch, pl, d, 1, status, sms, reinterpret_cast<cudaStream_t>(stream));
}
