/*
 * pagedattn.h -- C ABI of libpagedattn.so: paged-KV grouped-query attention
 * for Qwen3-style dense decoding on NVIDIA GB300 (sm_103a).
 *
 * Operations and the passages that define them:
 *  - pa_kv_write: "KV cache write" (decode) / "KV cache update" (prefill) in
 *    the "Qwen3-14B" pypto-lib doc, "Model structure, top down"; the slot
 *    formula blockId * blockSize + offset of ScatterKv in the "Qwen 3"
 *    TensorSharp doc, section 11 "Batched / paged forward".
 *  - pa_decode: the paged attention stage of decode_fwd ("Qwen3-14B",
 *    "decode_fwd"): vLLM ABI, token-major Q/O, flat K/V ordered
 *    [page, token, kv_head, dim]; K/V gathered per sequence from the block
 *    table and the sequence lengths ("Qwen 3", section 11).  Split across
 *    KV ranges (flash-decoding) and merged by pa_combine.
 *  - pa_decode_prologue: pa_qk_norm_rope_write and pa_decode as one kernel
 *    (decode_fwd's attention kernel with its in-kernel RoPE/QKV phase).
 *  - pa_decode_multi: the same causal attention for q_len new tokens per
 *    sequence (every chunk q_len long), run as B * q_len decode queries.
 *  - pa_kv_write_fp8 / pa_qk_norm_rope_write_fp8 / pa_decode_fp8 /
 *    pa_prefill_chunk_fp8: the same write, prologue, decode and prefill over
 *    an FP8 (e4m3) cache with per-KV-head scales.
 *  - pa_prefill_chunk: "KV cache update -> causal attention" of prefill_fwd
 *    ("Qwen3-14B", "prefill_fwd"), inputs packed token-major with
 *    T = sum(chunk_lens); full causal attention without window or sinks
 *    ("Qwen 3", 4.1 "Attention").
 *  - pa_combine: log-sum-exp merge of partial softmax states over disjoint
 *    key ranges (the split-K step of flash-decoding; not on the pages).
 *
 * Conventions shared by every entry point
 *  - Every tensor pointer is a DEVICE pointer owned by the caller; no call
 *    allocates device memory (pa_decode_noalloc's fixed scratch array is part
 *    of the loaded library).  Calls are asynchronous on `stream`
 *    (a cudaStream_t; NULL = the legacy default stream).
 *  - bf16 = IEEE bfloat16.  Layouts are dense row-major:
 *      q, out (decode)   [B, Hq, D]          (one query token per sequence)
 *      q, out (prefill)  [T, Hq, D]          (token-major, sequences in order)
 *      k_new, v_new      [T, Hkv, D]
 *      k_cache, v_cache  [num_pages, P, Hkv, D]
 *      block_table       int32 [B, max_pages_per_seq]
 *      context_lens      int32 [B]  tokens in the cache AFTER this step's write
 *      chunk_lens        int32 [B]  new tokens of each sequence this step
 *    with D = 128 (head_dim) and P = 128 (page_size).  New token j of
 *    sequence s sits at position context_lens[s] - chunk_lens[s] + j, in slot
 *    block_table[s][pos / P] * P + pos % P, and attends to keys 0..pos.
 *    Query head g uses KV head g / (Hq / Hkv).
 *  - Block-table entries past ceil(context_lens[s] / P) are never read (any
 *    value, e.g. -1, is fine there).  A referenced entry outside
 *    [0, num_pages), a negative length, chunk_lens[s] > context_lens[s] or
 *    context_lens[s] > max_pages_per_seq * P makes that sequence invalid: the
 *    kernels set a bit in *status (when status != NULL), write nothing to the
 *    cache for it and give it all-zero attention output.  They never trap.
 *  - context_lens[s] == 0 gives all-zero output rows (padding rows of a
 *    padded batch are expressed this way).
 *  - Return value: PA_OK, a negative PA_ERR_* found on the host before any
 *    launch (nothing was enqueued), or a positive cudaError_t from a launch.
 *  - Pointers passed to the tensor-memory-access (TMA) path -- k_cache and
 *    v_cache -- must be 16-byte aligned; q, out, k_new, v_new and workspace
 *    must be 16-byte aligned as well.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pa_stream_t; /* same type as cudaStream_t */

typedef struct pa_dims {
  int32_t num_seqs;          /* B, >= 0 (0 = nothing to do)                  */
  int32_t num_q_heads;       /* Hq, multiple of Hkv, Hq / Hkv <= 16          */
  int32_t num_kv_heads;      /* Hkv >= 1                                     */
  int32_t head_dim;          /* D, must be 128                               */
  int32_t page_size;         /* P, must be 128                               */
  int32_t num_pages;         /* pages in the pool, >= 1, num_pages*P < 2^31  */
  int32_t max_pages_per_seq; /* row length of block_table, >= 1              */
} pa_dims;

/* output element types */
#define PA_BF16 0
#define PA_F32 1

/* host-side argument errors (returned; nothing launched) */
#define PA_OK 0
#define PA_ERR_NULL_POINTER (-1)
#define PA_ERR_HEAD_DIM (-2)
#define PA_ERR_PAGE_SIZE (-3)
#define PA_ERR_HEADS (-4)
#define PA_ERR_DIMS (-5)
#define PA_ERR_ALIGNMENT (-6)
#define PA_ERR_OUT_DTYPE (-7)
#define PA_ERR_WORKSPACE (-8)
#define PA_ERR_SPLITS (-9)
#define PA_ERR_TOO_MANY_SEQS (-10)
#define PA_ERR_TENSOR_MAP (-11)
#define PA_ERR_NO_DEVICE (-12)
#define PA_ERR_NOALLOC_TOO_LARGE (-13)

/* device-side status bits OR-ed into *status */
#define PA_STATUS_BAD_PAGE 1    /* referenced block-table entry out of range */
#define PA_STATUS_BAD_LENGTH 2  /* inconsistent context/chunk lengths        */
#define PA_STATUS_BAD_TOKENS 4  /* sum(chunk_lens) != num_tokens             */
#define PA_STATUS_TIMEOUT 8     /* a bounded wait inside a kernel gave up    */
#define PA_STATUS_Q_RANGE 16    /* FP8 cache: a q element is not finite     */

/* Largest batch accepted by the calls that take chunk_lens (the per-sequence
 * token offsets are built in shared memory). */
#define PA_MAX_CHUNKED_SEQS 16384

/* Largest Hq + 2 Hkv that pa_qk_norm_rope_write takes. */
#define PA_MAX_PROLOGUE_HEADS 384

/* num_splits value for pa_decode's page-balanced schedule (see pa_decode). */
#define PA_SPLITS_BALANCED (-1)
/* Largest batch the page-balanced schedule takes. */
#define PA_BALANCED_MAX_SEQS 512

/*
 * pa_kv_write -- copy the new tokens' K and V rows into their cache slots.
 *   k_new, v_new   bf16 [num_tokens, Hkv, D], token-major in sequence order
 *   k_cache,v_cache bf16 [num_pages, P, Hkv, D], written in place
 *   block_table, context_lens: as above (context_lens counts the new tokens)
 *   chunk_lens     int32 [B] new tokens per sequence, or NULL for decode
 *                  (one token per sequence, num_tokens must equal B)
 *   status         device int32, may be NULL; bits PA_STATUS_* are OR-ed in
 * A bit copy: every written byte equals the source byte; no other cache byte
 * changes.  Two sequences must not write the same slot in one call.
 */
int pa_kv_write(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                const int32_t* block_table, const int32_t* context_lens,
                const int32_t* chunk_lens, int32_t num_tokens, pa_dims dims,
                int32_t* status, pa_stream_t stream);

/*
 * pa_qk_norm_rope_write -- the prologue of decode and prefill: per-head
 * RMSNorm of Q and K, NeoX rotary embedding at each new token's position, and
 * the KV cache write, fused in one pass.  "Qwen 3" (TensorSharp model doc),
 * section 3 "Forward graph" (per-head RMSNorm(Q) / RMSNorm(K) with
 * attn_q_norm / attn_k_norm, RoPE_NeoX at the tokens' positions, Q times
 * 1/sqrt(headDim), (K, V) appended to the cache), section 4.1 (QK-norm over
 * each head's headDim values; NeoX RoPE from rope.freq_base and rope.scale),
 * section 4.3 (epsilon); "Qwen3-14B" (pypto-lib), "Model structure, top down"
 * (decode_fwd: Q/K norm -> RoPE -> KV cache write; FP32 RMSNorm weights).
 *   qkv            bf16 [num_tokens, (Hq + 2 Hkv) * D]: the fused projection's
 *                  rows, [Hq query heads | Hkv key heads | Hkv value heads]
 *   q_norm_w, k_norm_w  float32 [D], the per-head RMSNorm weights
 *   eps            RMSNorm epsilon: y = x / sqrt(mean(x^2) + eps) * w
 *   rope_base, rope_scale  pair (i, i + D/2) turns by pos * base^(-2i/D) / scale
 *   q_scale        multiplies Q after RoPE (1/sqrt(D) to fold the softmax scale
 *                  into Q, then call pa_decode with scale 1; or 1)
 *   q_out          bf16 [num_tokens, Hq, D], the input of pa_decode /
 *                  pa_prefill_chunk; rows of an invalid sequence are zero
 *   k_cache, v_cache, block_table, context_lens, chunk_lens, num_tokens,
 *   status: exactly as pa_kv_write (K is written normed and rotated, rounded
 *   to bf16; V bit for bit).  Positions are context_lens[s] - chunk_lens[s] + j.
 * Returns PA_ERR_DIMS for eps < 0, rope_base <= 0, rope_scale <= 0 or a
 * non-finite value, PA_ERR_HEADS when Hq + 2 Hkv > PA_MAX_PROLOGUE_HEADS (a
 * token's row is staged whole in shared memory); every pointer must be
 * 16-byte aligned.
 */
int pa_qk_norm_rope_write(const void* qkv, const float* q_norm_w, const float* k_norm_w,
                          float eps, float rope_base, float rope_scale, float q_scale,
                          void* q_out, void* k_cache, void* v_cache,
                          const int32_t* block_table, const int32_t* context_lens,
                          const int32_t* chunk_lens, int32_t num_tokens, pa_dims dims,
                          int32_t* status, pa_stream_t stream);

/*
 * pa_decode -- single-token paged GQA attention, one query token per sequence.
 *   q              bf16 [B, Hq, D]
 *   scale          multiplies every score q.k (1/sqrt(D) for Qwen3)
 *   out            [B, Hq, D], element type out_dtype (PA_BF16 or PA_F32)
 *   workspace      device scratch for split partials, at least
 *                  pa_decode_workspace_size(dims, num_splits) bytes; may be
 *                  NULL when that size is 0.  Caller-owned; contents need no
 *                  initialisation and are overwritten.
 *   num_splits     the work schedule:
 *                  1..max_pages_per_seq: fixed splits -- each sequence's pages
 *                    are divided into that many equal KV ranges, dealt to the
 *                    SMs round-robin.  With one split the kernel writes `out`
 *                    directly; otherwise it writes partials to the workspace
 *                    and runs the pa_combine kernel.
 *                  PA_SPLITS_BALANCED: page-balanced -- the SMs form groups
 *                    of one SM per KV head; the sequences' pages, laid end to
 *                    end, are divided evenly among the groups, so every SM
 *                    reads the same number of pages and the SMs of a group
 *                    read the same pages together.  The few sequences cut
 *                    between two groups are merged by a combine kernel.  This
 *                    balances ragged batches.  B <= PA_BALANCED_MAX_SEQS and
 *                    at least two groups must fit on the device.
 *                  0: the library chooses from the shape and the device's SM
 *                    count (pa_decode_auto_splits).
 * The result depends only on logical positions, never on which physical
 * pages hold them: the same inputs under a permuted pool and rewritten block
 * table give bit-identical output.
 */
int pa_decode(const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_table, const int32_t* context_lens, float scale,
              void* out, int32_t out_dtype, void* workspace, size_t workspace_bytes,
              int32_t num_splits, pa_dims dims, int32_t* status, pa_stream_t stream);

/* Workspace bytes pa_decode needs for num_splits (0 = the automatic choice on
 * the current device).  Returns 0 when no workspace is needed, and
 * (size_t)-1 for invalid dims. */
size_t pa_decode_workspace_size(pa_dims dims, int32_t num_splits);

/* The schedule pa_decode uses for num_splits == 0 on the current device: a
 * split count >= 1, or 0 for the page-balanced schedule; a negative PA_ERR_*
 * for invalid dims. */
int32_t pa_decode_auto_splits(pa_dims dims);

/* Largest q_len pa_decode_multi takes. */
#define PA_MAX_Q_LEN 16

/*
 * pa_decode_multi -- multi-token decode (speculative-decoding verification,
 * multi-token prediction): q_len new tokens per sequence, each attending
 * causally over the paged cache.  This is the causal attention step of
 * "prefill_fwd" ("Qwen3-14B", pypto-lib doc) with every chunk q_len long,
 * run on the decode kernel: token j of sequence s sits at position
 * context_lens[s] - q_len + j and attends to keys 0 .. that position.  Each
 * decode work item stacks (token, query head) pairs of one KV head -- up to 32
 * of them -- in the columns of its tensor-core products, so a K/V page is read
 * once for all the tokens it serves.
 *   q              bf16 [B * q_len, Hq, D], token-major in sequence order
 *                  (the packing of pa_prefill_chunk with chunk_lens = q_len)
 *   q_len          1 .. PA_MAX_Q_LEN; the new tokens must already be in the
 *                  cache (pa_kv_write with chunk_lens = q_len)
 *   out            [B * q_len, Hq, D], element type out_dtype
 *   workspace      at least pa_decode_multi_workspace_size(dims, q_len,
 *                  num_splits) bytes (caller-owned, no initialisation)
 *   num_splits     as pa_decode (the balanced schedule needs
 *                  B <= PA_BALANCED_MAX_SEQS)
 *   dims.num_seqs  B (sequences; the block table has B rows)
 * A sequence with 0 < context_lens[s] < q_len is invalid (status bit
 * PA_STATUS_BAD_LENGTH, zero output); context_lens[s] == 0 gives zero rows.
 * q_len == 1 is exactly pa_decode.  Returns PA_ERR_DIMS for q_len out of range.
 */
int pa_decode_multi(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_table, const int32_t* context_lens, int32_t q_len,
                    float scale, void* out, int32_t out_dtype, void* workspace,
                    size_t workspace_bytes, int32_t num_splits, pa_dims dims,
                    int32_t* status, pa_stream_t stream);

/* Workspace bytes pa_decode_multi (and pa_decode_fp8) need; (size_t)-1 for
 * invalid arguments. */
size_t pa_decode_multi_workspace_size(pa_dims dims, int32_t q_len, int32_t num_splits);

/*
 * FP8 KV cache: the "fp8_e4m3" KV cache dtype (SGLang, as quoted in the
 * "Qwen4-Exp QSA trafia na Ascend..." blog; a quantized KV dtype is also the
 * --kv-cache-dtype option of the "Qwen 3" TensorSharp doc, section 11).
 * k_cache, v_cache  uint8 [num_pages, P, Hkv, D] e4m3fn codes (sign, 4
 *                   exponent bits with bias 7, 3 mantissa bits; no infinities;
 *                   largest finite 448) -- half the bytes of the bf16 cache
 * k_scale, v_scale  float32 [Hkv] device arrays: a cached code c of KV head h
 *                   means value(c) * scale[h]
 */

/*
 * pa_kv_write_fp8 -- pa_kv_write into an FP8 cache: element d of KV head h is
 * stored as the e4m3 code of x / scale[h] (the FP32 quotient, rounded to
 * nearest with ties to even, saturating at +-448; NaN stays NaN).  Slots,
 * validity rules and status bits are those of pa_kv_write.  k_scale and
 * v_scale must be non-null and 4-byte aligned.
 */
int pa_kv_write_fp8(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                    const float* k_scale, const float* v_scale, const int32_t* block_table,
                    const int32_t* context_lens, const int32_t* chunk_lens,
                    int32_t num_tokens, pa_dims dims, int32_t* status, pa_stream_t stream);

/*
 * pa_qk_norm_rope_write_fp8 -- pa_qk_norm_rope_write into an FP8 cache: the
 * decode / prefill prologue ("Qwen 3" TensorSharp doc, section 3; "Qwen3-14B"
 * pypto-lib doc, decode_fwd) writing an "fp8_e4m3" KV cache ("Qwen4-Exp QSA"
 * blog, DGX Spark note; "Qwen 3" section 11, --kv-cache-dtype).  Each stored
 * row is quantized as pa_kv_write_fp8 quantizes a bf16 row: K normed, rotated
 * and rounded to bf16 as pa_qk_norm_rope_write stores it, V as given, element
 * d of KV head h divided by k_scale[h] / v_scale[h] (FP32 quotient) and
 * rounded to the nearest e4m3 code (ties to even, saturating at +-448).  The
 * cache bytes equal those of pa_qk_norm_rope_write into a bf16 cache followed
 * by pa_kv_write_fp8 of the rows it wrote; q_out, validity rules, status bits
 * and the other arguments are those of pa_qk_norm_rope_write.
 *   k_cache, v_cache  uint8 e4m3 codes [num_pages, P, Hkv, D], written in place
 *   k_scale, v_scale  float32 [Hkv] device arrays, non-null and 4-byte aligned
 */
int pa_qk_norm_rope_write_fp8(const void* qkv, const float* q_norm_w, const float* k_norm_w,
                              float eps, float rope_base, float rope_scale, float q_scale,
                              void* q_out, void* k_cache, void* v_cache, const float* k_scale,
                              const float* v_scale, const int32_t* block_table,
                              const int32_t* context_lens, const int32_t* chunk_lens,
                              int32_t num_tokens, pa_dims dims, int32_t* status,
                              pa_stream_t stream);

/*
 * pa_decode_prologue -- the decode step with its prologue in the attention
 * kernel: "Qwen3-14B" (pypto-lib), "Model structure, top down" (decode_fwd:
 * Q/K norm -> RoPE -> KV cache write -> paged attention; the CCE attention
 * kernel there runs the RoPE/QKV step as its in-kernel phase 0).  For one
 * new token per sequence: the query heads are normed, rotated and scaled from
 * the fused projection row inside the kernel (never written out), the new
 * token's K row (normed, rotated) and V row are written to its cache slot,
 * and the token attends to its whole context, new token included.  The cache
 * bytes and `out` equal those of pa_qk_norm_rope_write (chunk_lens NULL)
 * followed by pa_decode with the same arguments, bit for bit, and so do the
 * status bits (context_lens[s] == 0 flags PA_STATUS_BAD_LENGTH, as the
 * prologue flags a token without a position, and gives a zero row).
 *   qkv, q_norm_w, k_norm_w, eps, rope_base, rope_scale, q_scale: as
 *                  pa_qk_norm_rope_write, num_tokens = num_seqs
 *   k_cache, v_cache, block_table, context_lens, scale, out, out_dtype,
 *   workspace, num_splits, status: as pa_decode (the same workspace size)
 * Returns PA_ERR_HEADS when Hq / Hkv > 16; otherwise the checks of
 * pa_qk_norm_rope_write and pa_decode.
 */
int pa_decode_prologue(const void* qkv, const float* q_norm_w, const float* k_norm_w, float eps,
                       float rope_base, float rope_scale, float q_scale, void* k_cache,
                       void* v_cache, const int32_t* block_table, const int32_t* context_lens,
                       float scale, void* out, int32_t out_dtype, void* workspace,
                       size_t workspace_bytes, int32_t num_splits, pa_dims dims,
                       int32_t* status, pa_stream_t stream);

/*
 * pa_decode_fp8 -- pa_decode_multi over an FP8 cache (q_len = 1: single-token
 * decode).  The K/V pages are read as e4m3 (half the bytes).  q . K runs on
 * the e4m3 K codes themselves: each query row, times a power of two x that
 * brings its work item's largest |q| into [128, 256), is split into two e4m3
 * rows hi + lo, which equal it exactly for every element of magnitude at
 * least 2^-10 of that largest (smaller ones are off by at most 2^-10 / x), so
 * q may take any finite bf16 value; a non-finite q element sets
 * PA_STATUS_Q_RANGE and makes its item's output NaN.  V is converted on the
 * chip to F16, which holds every e4m3 value exactly, and P is rounded to F16
 * for the P.V product.  The scores are q . K * k_scale[h] * scale and the
 * output is multiplied by v_scale[h].  Arguments, schedules, workspace
 * (pa_decode_multi_workspace_size) and status bits as pa_decode_multi.
 */
int pa_decode_fp8(const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                  const float* v_scale, const int32_t* block_table,
                  const int32_t* context_lens, int32_t q_len, float scale, void* out,
                  int32_t out_dtype, void* workspace, size_t workspace_bytes,
                  int32_t num_splits, pa_dims dims, int32_t* status, pa_stream_t stream);

/*
 * pa_prefill_chunk -- causal attention of a packed chunk of new tokens over
 * the paged cache (prior context plus the chunk itself, which pa_kv_write
 * must already have written).
 *   q              bf16 [num_tokens, Hq, D], token-major in sequence order
 *   chunk_lens     int32 [B], sum must equal num_tokens (B <= PA_MAX_CHUNKED_SEQS)
 *   out            [num_tokens, Hq, D], element type out_dtype
 * Token j of sequence s attends to keys 0..context_lens[s]-chunk_lens[s]+j.
 */
int pa_prefill_chunk(const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_table, const int32_t* context_lens,
                     const int32_t* chunk_lens, int32_t num_tokens, float scale,
                     void* out, int32_t out_dtype, pa_dims dims, int32_t* status,
                     pa_stream_t stream);

/*
 * pa_prefill_chunk_fp8 -- pa_prefill_chunk over an FP8 (e4m3) cache, the
 * prefill step ("Qwen3-14B" pypto-lib doc, prefill_fwd: KV cache update, then
 * causal attention) with the "fp8_e4m3" KV cache dtype the SGLang launch in
 * the "Qwen4-Exp QSA..." blog selects.  The chunk's own K/V must already be
 * in the cache (pa_kv_write_fp8).  q . K runs on the e4m3 K codes as in
 * pa_decode_fp8, with each query row split into e4m3 hi + lo after scaling by
 * a power of two of its own (exact for every element of magnitude at least
 * 2^-10 of the row's largest; any finite bf16 q; a non-finite element sets
 * PA_STATUS_Q_RANGE and makes its row NaN); V is converted on the chip to
 * F16, which holds every e4m3 value exactly, and P is rounded to F16 for the
 * P.V product.  The
 * scores are q . K * k_scale[h] * scale and the output is multiplied by
 * v_scale[h].  Arguments, limits, status bits and errors as pa_prefill_chunk;
 * k_scale and v_scale (float32 [Hkv], device) must be non-null
 * (PA_ERR_NULL_POINTER) and 4-byte aligned (PA_ERR_ALIGNMENT).
 */
int pa_prefill_chunk_fp8(const void* q, const void* k_cache, const void* v_cache,
                         const float* k_scale, const float* v_scale,
                         const int32_t* block_table, const int32_t* context_lens,
                         const int32_t* chunk_lens, int32_t num_tokens, float scale,
                         void* out, int32_t out_dtype, pa_dims dims, int32_t* status,
                         pa_stream_t stream);

/*
 * pa_combine -- merge num_splits partial attention states per (sequence, head).
 *   part_o         float32 [B, Hq, num_splits, D]; state i normalised by its own
 *                  softmax sum
 *   part_lse       float32 [B, Hq, num_splits]; natural-log sum of exp(score)
 *                  over state i's keys, -inf for a state with no keys
 *   out            [B, Hq, D], out_dtype
 * out = sum_i exp(lse_i - LSE) * o_i with LSE = log(sum_i exp(lse_i)); a row
 * whose states are all -inf is zero; a row with any +inf lse (the marker
 * pa_decode writes for an invalid sequence) is zero.  Uses num_seqs,
 * num_q_heads and head_dim of dims.
 */
int pa_combine(const float* part_o, const float* part_lse, int32_t num_splits, void* out,
               int32_t out_dtype, pa_dims dims, pa_stream_t stream);

/* Largest k pa_topk takes (the pages' fixed candidate capacity). */
#define PA_TOPK_MAX_K 32

/*
 * pa_topk -- exact top-k of each row of logits: the sampling candidates.
 * pypto-serving PR #77 ("Qwen3-14B device top-k"), "Exactness Design": an
 * exact Top-32 of the full-vocabulary logits (151936 real entries for
 * Qwen3-14B), merged hierarchically from exact per-group Top-k sets, returning
 * candidate values and token IDs; checked against torch.topk.
 *   logits         float32, row r at logits + r * row_stride, its first vocab
 *                  entries used (row_stride >= vocab; 4-byte aligned)
 *   k              1 .. PA_TOPK_MAX_K, <= vocab
 *   out_values     float32 [rows, k], out_indices int32 [rows, k]: the k
 *                  largest entries, larger first; NaN ranks above +inf; equal
 *                  values (including -0 and +0) by smaller index.  A value is the
 *                  logit as given.
 *   workspace      device scratch of pa_topk_workspace_size(rows, vocab, k)
 *                  bytes (16-byte aligned), contents need no initialisation
 * Returns PA_ERR_DIMS for an unsupported k / vocab / row_stride.
 */
int pa_topk(const float* logits, int64_t row_stride, int32_t rows, int32_t vocab, int32_t k,
            float* out_values, int32_t* out_indices, void* workspace, size_t workspace_bytes,
            pa_stream_t stream);

/* Workspace bytes pa_topk needs on the current device, (size_t)-1 for invalid
 * arguments. */
size_t pa_topk_workspace_size(int32_t rows, int32_t vocab, int32_t k);

/* Size of the device array pa_decode_noalloc keeps its split partials in. */
#define PA_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/*
 * pa_decode_noalloc -- pa_decode for callers that cannot allocate device
 * memory.  (This entry point has no counterpart on the source pages; it
 * exists for integration.)  Some callers are handed their input and output
 * buffers by a host framework that owns every device allocation -- an engine
 * plugin, or a C host with no device allocator of its own -- and others must
 * not call cudaMalloc on a latency-critical path, where it can synchronise
 * the device.  Such callers cannot provide pa_decode's workspace.
 *
 * Same arguments, layouts, results and status handling as pa_decode, without
 * workspace / workspace_bytes.  The split partials go to one device array of
 * PA_NOALLOC_SCRATCH_BYTES (16 MiB) inside the library; every GPU that loads
 * the library holds that array until the process exits.  A call whose split
 * count (num_splits, or the automatic choice for 0) needs more scratch than
 * that -- (B * Hq * splits * 516 bytes, rounded up; the page-balanced
 * schedule needs about 5 MB on 152 SMs) -- returns PA_ERR_NOALLOC_TOO_LARGE without
 * launching; num_splits = 1 needs none.
 *
 * Setup: the first call made with a given device current looks up the
 * array's device address on that device (cudaGetSymbolAddress) and caches it;
 * make that first call before any stream capture.  Nothing is allocated, by
 * this function or by anything it calls.
 *
 * Sharing: all calls on a device use the same array, which keeps whatever the
 * last call left in it.  Nothing in it needs to start at zero -- every partial
 * the combine step reads is written earlier in the same call -- but calls
 * that can overlap on the GPU (different streams, or different host threads
 * without ordering) race on the array and corrupt each other's results:
 * order them on one stream, or use pa_decode with separate workspaces.
 */
int pa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_table, const int32_t* context_lens, float scale,
                      void* out, int32_t out_dtype, int32_t num_splits, pa_dims dims,
                      int32_t* status, pa_stream_t stream);

/* Work items (sequence, pair of 128-token query tiles, query head) that each
 * CTA pair of a pa_prefill_chunk launch schedules longest-first; launches
 * with more than PA_PREFILL_SCHEDULE_ITEMS x pa_prefill_pairs() items deal
 * them round-robin instead. */
#define PA_PREFILL_SCHEDULE_ITEMS 64

/*
 * pa_prefill_pairs -- CTA pairs (clusters of two CTAs on two SMs) that a
 * pa_prefill_chunk launch uses at most on the current device: the pairs that
 * fit on the GPU at once.  Returns the count (>= 1), PA_ERR_NO_DEVICE, or a
 * positive CUDA error.
 */
int32_t pa_prefill_pairs(void);

/*
 * pa_wait_selftest -- run the kernels' bounded-wait failure path once, on
 * purpose and without a fault.  The only device failure the pages report is a
 * timeout (the "507018" timeout of oversized task-graph prototypes in the
 * pypto-serving top-k PR, "Exactness Design"); here every mbarrier wait inside
 * a kernel gives up after a limit, sets PA_STATUS_TIMEOUT, drains the copies
 * it has in flight and returns, so the context stays usable.
 *
 * Launches one CTA of 64 threads on `stream` that waits, with the same wait
 * routines (one warp-uniform, one single-thread), on a shared-memory mbarrier
 * that nothing arrives on, giving up after limit_us microseconds (1 ..
 * 5,000,000; the attention kernels use 2 s).  No bulk copy is in flight.
 *   status   device int32, required: PA_STATUS_TIMEOUT is OR-ed in when the
 *            waits give up (the expected outcome); PA_STATUS_BAD_LENGTH too if
 *            a wait ever reported a phase that never completed.
 * Returns PA_ERR_DIMS for a limit out of range, PA_ERR_NULL_POINTER for a NULL
 * status, or a positive CUDA launch error.
 */
int pa_wait_selftest(uint32_t limit_us, int32_t* status, pa_stream_t stream);

/* Human-readable text for a return code (negative PA_ERR_* or positive CUDA
 * error).  Never NULL; the string is static. */
const char* pa_status_string(int32_t code);

/* ABI version of this header (major * 100 + minor). */
int32_t pa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
