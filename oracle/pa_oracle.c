/*
 * Paged-KV GQA attention oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU implementation of what the paged
 * attention path computes, in double precision.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may load this file's
 * library; the product path never does.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * Sources (page title, section):
 *  - "Qwen3-14B" (pypto-lib model doc), "Model structure, top down":
 *    decode_fwd writes the new token into the KV cache and then runs paged
 *    attention; prefill_fwd does "KV cache update -> causal attention" over
 *    token-major packed inputs (T = sum(chunk_lens)).  "Deployment
 *    configuration": 128-token pages.  The attention ABI: Q/O are token-major
 *    (TND), the flat paged K/V buffers are ordered [page, token, kv_head, dim].
 *  - "Qwen 3" (TensorSharp model doc), section 11 "Batched / paged forward":
 *    K/V are scattered to slot blockId*blockSize + offset and gathered per
 *    sequence from the block tables and sequence lengths; section 3 "Forward
 *    graph" and 4.1 "Attention": full causal GQA, no window, no sinks, the
 *    softmax scale 1/sqrt(headDim) folded into the scores.
 *  - "Qwen4-Exp QSA trafia na Ascend..." (orcarouter blog), first section's
 *    size-limit bullet: -1 padding is not a valid slot, fully masked rows
 *    produce zero output.
 *
 * Readings where the pages are silent:
 *  - query head g reads KV head g / (Hq/Hkv) (contiguous groups);
 *  - context_lens[s] counts tokens AFTER the write; chunk_lens[s] new tokens;
 *    new token j of sequence s sits at position context_lens[s]-chunk_lens[s]+j
 *    and sees keys 0..position (decode: chunk_lens == NULL means 1 each);
 *  - scores are multiplied by the caller's `scale`;
 *  - an empty context, or any referenced block-table entry outside
 *    [0, num_pages), or lengths that do not fit the block table, give an
 *    all-zero output for every row of that sequence.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bfloat16 bits -> double, exactly (a bf16 is the top half of an IEEE float). */
static double bf16_to_f64(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* ---------------------------------------------------------------------------
 * FP8 KV cache ("fp8_e4m3" KV cache in the SGLang measurement of the
 * "Qwen4-Exp QSA trafia na Ascend..." blog; a quantized KV dtype is also the
 * --kv-cache-dtype option of the "Qwen 3" TensorSharp doc, section 11).
 * Readings: e4m3 is the e4m3fn encoding (sign, 4
 * exponent bits with bias 7, 3 mantissa bits; no infinities; S.1111.111 is
 * NaN; largest finite 448); every KV head h has one FP32 scale for K and one
 * for V; a cached value means code_value * scale; writing divides the bf16
 * value by the scale in FP32 and rounds that quotient to the nearest e4m3
 * value, ties to the even code, saturating at +-448.
 * ------------------------------------------------------------------------- */

/* Value of e4m3 code c (NaN for the two NaN codes). */
double oracle_e4m3_decode(uint8_t c) {
  int sgn = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  double v = e == 0 ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
  return sgn ? -v : v;
}

/* Nearest e4m3 code to x: the finite code of least distance, the even code
 * on a tie; |x| >= 448 (infinity too) gives +-448, NaN a NaN code; the sign
 * of x (zero included) is kept. */
uint8_t oracle_e4m3_encode(float x) {
  uint8_t sgn = signbit(x) ? 0x80 : 0;
  if (isnan(x)) return sgn | 0x7F;
  double a = fabs((double)x);
  if (a >= 448.0) return sgn | 0x7E;
  int best = 0;
  double bd = INFINITY;
  for (int c = 0; c <= 0x7E; ++c) {
    double d = fabs(oracle_e4m3_decode((uint8_t)c) - a);
    if (d < bd || (d == bd && (c & 1) == 0)) {
      bd = d;
      best = c;
    }
  }
  return sgn | (uint8_t)best;
}

/* Array forms for the Python side. */
void oracle_e4m3_encode_array(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(x[i]);
}
void oracle_e4m3_decode_array(const uint8_t* c, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(c[i]);
}

/* Cache element formats: bf16 values, or e4m3 codes times a per-head scale. */
enum { KV_BF16 = 0, KV_E4M3 = 1 };

static double kv_value(const void* cache, int64_t idx, int fmt, double scale) {
  if (fmt == KV_BF16) return bf16_to_f64(((const uint16_t*)cache)[idx]);
  return oracle_e4m3_decode(((const uint8_t*)cache)[idx]) * scale;
}

/* Validity of sequence s: lengths consistent and every page it references in
 * range.  Returns 1 when the sequence may be attended/written. */
static int seq_valid(const int32_t* block_table, const int32_t* context_lens,
                     const int32_t* chunk_lens, int s, int page_size,
                     int num_pages, int max_pages_per_seq) {
  int64_t ctx = context_lens[s];
  int64_t n = chunk_lens ? chunk_lens[s] : 1;
  if (ctx < 0 || n < 0 || n > ctx) return 0;
  if (ctx > (int64_t)max_pages_per_seq * page_size) return 0;
  int64_t used = (ctx + page_size - 1) / page_size;
  for (int64_t i = 0; i < used; ++i) {
    int32_t p = block_table[(int64_t)s * max_pages_per_seq + i];
    if (p < 0 || p >= num_pages) return 0;
  }
  return 1;
}

/*
 * KV write ("KV cache write" / "KV cache update" in the Qwen3-14B doc;
 * ScatterKv in the TensorSharp doc, section 11): for new token j of sequence
 * s, position pos = ctx - n + j, slot = block_table[s][pos / P] * P + pos % P;
 * copy the token's [Hkv, D] K and V rows into the cache at that slot.  A byte
 * copy: no arithmetic on the values.  Tokens of an invalid sequence are not
 * written, and neither are tokens past the num_tokens rows the caller passed.
 * Returns the number of sequences skipped as invalid.
 */
int oracle_kv_write(const uint16_t* k_new, const uint16_t* v_new,
                    uint16_t* k_cache, uint16_t* v_cache,
                    const int32_t* block_table, const int32_t* context_lens,
                    const int32_t* chunk_lens, int64_t num_tokens, int num_seqs,
                    int num_kv_heads, int head_dim, int page_size, int num_pages,
                    int max_pages_per_seq) {
  const int64_t row = (int64_t)num_kv_heads * head_dim; /* elements per token */
  int64_t token = 0;
  int skipped = 0;
  for (int s = 0; s < num_seqs; ++s) {
    int64_t n = chunk_lens ? chunk_lens[s] : 1;
    if (!seq_valid(block_table, context_lens, chunk_lens, s, page_size,
                   num_pages, max_pages_per_seq)) {
      ++skipped;
      token += n > 0 ? n : 0;
      continue;
    }
    int64_t ctx = context_lens[s];
    for (int64_t j = 0; j < n && token < num_tokens; ++j, ++token) {
      int64_t pos = ctx - n + j;
      int64_t page = block_table[(int64_t)s * max_pages_per_seq + pos / page_size];
      int64_t slot = page * page_size + pos % page_size;
      memcpy(k_cache + slot * row, k_new + token * row, (size_t)row * 2);
      memcpy(v_cache + slot * row, v_new + token * row, (size_t)row * 2);
    }
  }
  return skipped;
}

/*
 * FP8 KV write: the same slots as oracle_kv_write; element d of KV head h of a
 * token is stored as the e4m3 code of (float)x / scale[h] (an FP32 quotient).
 * Returns the number of sequences skipped as invalid.
 */
int oracle_kv_write_fp8(const uint16_t* k_new, const uint16_t* v_new, uint8_t* k_cache,
                        uint8_t* v_cache, const float* k_scale, const float* v_scale,
                        const int32_t* block_table, const int32_t* context_lens,
                        const int32_t* chunk_lens, int64_t num_tokens, int num_seqs,
                        int num_kv_heads, int head_dim, int page_size, int num_pages,
                        int max_pages_per_seq) {
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  int64_t token = 0;
  int skipped = 0;
  for (int s = 0; s < num_seqs; ++s) {
    int64_t n = chunk_lens ? chunk_lens[s] : 1;
    if (!seq_valid(block_table, context_lens, chunk_lens, s, page_size, num_pages,
                   max_pages_per_seq)) {
      ++skipped;
      token += n > 0 ? n : 0;
      continue;
    }
    int64_t ctx = context_lens[s];
    for (int64_t j = 0; j < n && token < num_tokens; ++j, ++token) {
      int64_t pos = ctx - n + j;
      int64_t page = block_table[(int64_t)s * max_pages_per_seq + pos / page_size];
      int64_t slot = page * page_size + pos % page_size;
      for (int h = 0; h < num_kv_heads; ++h)
        for (int d = 0; d < head_dim; ++d) {
          int64_t i = (int64_t)h * head_dim + d;
          float kq = (float)bf16_to_f64(k_new[token * row + i]) / k_scale[h];
          float vq = (float)bf16_to_f64(v_new[token * row + i]) / v_scale[h];
          k_cache[slot * row + i] = oracle_e4m3_encode(kq);
          v_cache[slot * row + i] = oracle_e4m3_encode(vq);
        }
    }
  }
  return skipped;
}

/*
 * Dense softmax attention of one query over n keys (steps 2-3 of the
 * definition): x_t = scale * <q, K_t>, m = max_t x_t, w_t = exp(x_t - m),
 * out = sum_t w_t V_t / sum_t w_t.  Also returns lse = m + log(sum_t w_t), the
 * natural-log normaliser of this key set (used to pin the split combine).
 * n == 0 gives out = 0 and lse = -inf.
 */
void oracle_dense_attention(const double* q, const double* K, const double* V,
                            int64_t n, int head_dim, double scale, double* out,
                            double* lse, double* x /* scratch, n */) {
  for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
  if (n <= 0) { if (lse) *lse = -INFINITY; return; }
  double m = -INFINITY;
  for (int64_t t = 0; t < n; ++t) {
    double dot = 0.0;
    for (int d = 0; d < head_dim; ++d) dot += q[d] * K[t * head_dim + d];
    x[t] = scale * dot;
    if (x[t] > m) m = x[t];
  }
  double denom = 0.0;
  for (int64_t t = 0; t < n; ++t) {
    double w = exp(x[t] - m);
    denom += w;
    for (int d = 0; d < head_dim; ++d) out[d] += w * V[t * head_dim + d];
  }
  for (int d = 0; d < head_dim; ++d) out[d] /= denom;
  if (lse) *lse = m + log(denom);
}

/*
 * One (token, query head) row: step 1 of the definition gathers K_t, V_t for
 * t = 0..pos through the block table (slot = page * P + t % P) into dense
 * double buffers, then the dense attention above.
 */
static void attend_row(const uint16_t* qrow, const void* k_cache,
                       const void* v_cache, int fmt, double ks, double vs,
                       const int32_t* bt_row, int64_t pos, int kv_head, int num_kv_heads,
                       int head_dim, int page_size, double scale, double* out,
                       double* qd, double* K, double* V, double* x) {
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  int64_t nkeys = pos + 1;
  for (int d = 0; d < head_dim; ++d) qd[d] = bf16_to_f64(qrow[d]);
  for (int64_t t = 0; t < nkeys; ++t) {
    int64_t slot = (int64_t)bt_row[t / page_size] * page_size + t % page_size;
    int64_t base = slot * row + (int64_t)kv_head * head_dim;
    for (int d = 0; d < head_dim; ++d) {
      K[t * head_dim + d] = kv_value(k_cache, base + d, fmt, ks);
      V[t * head_dim + d] = kv_value(v_cache, base + d, fmt, vs);
    }
  }
  oracle_dense_attention(qd, K, V, nkeys, head_dim, scale, out, NULL, x);
}

/*
 * Attention over the paged cache for packed token-major queries.
 *   q:   [T, Hq, D] bf16 bits, T = sum(chunk_lens) (decode: chunk_lens == NULL,
 *        T = num_seqs, one token per sequence)
 *   out: [nrows, D] doubles; row r is (token, head) = rows[r] / Hq, rows[r] % Hq,
 *        or every row in order when rows == NULL (nrows must then be T*Hq).
 * Returns 0, or -1 if a requested row index is out of range.
 */
static int attention_impl(const uint16_t* q, const void* k_cache, const void* v_cache,
                          int fmt, const float* k_scale, const float* v_scale,
                          const int32_t* block_table, const int32_t* context_lens,
                          const int32_t* chunk_lens, int num_seqs, int num_q_heads,
                          int num_kv_heads, int head_dim, int page_size, int num_pages,
                          int max_pages_per_seq, double scale, const int64_t* rows,
                          int64_t nrows, double* out, int num_threads) {
  /* token -> (sequence, index within its chunk) */
  int64_t T = 0;
  for (int s = 0; s < num_seqs; ++s) T += chunk_lens ? (chunk_lens[s] > 0 ? chunk_lens[s] : 0) : 1;
  int32_t* tok_seq = (int32_t*)malloc(sizeof(int32_t) * (T > 0 ? T : 1));
  int64_t* tok_j = (int64_t*)malloc(sizeof(int64_t) * (T > 0 ? T : 1));
  int64_t maxctx = 1;
  {
    int64_t t = 0;
    for (int s = 0; s < num_seqs; ++s) {
      int64_t n = chunk_lens ? chunk_lens[s] : 1;
      for (int64_t j = 0; j < n; ++j, ++t) { tok_seq[t] = s; tok_j[t] = j; }
      if (context_lens[s] > maxctx) maxctx = context_lens[s];
    }
  }
  const int group = num_q_heads / num_kv_heads;
  int64_t total = rows ? nrows : T * num_q_heads;
  int bad = 0;
  if (!rows && nrows != T * num_q_heads) bad = 1;
  if (rows)
    for (int64_t r = 0; r < nrows; ++r)
      if (rows[r] < 0 || rows[r] >= T * num_q_heads) bad = 1;
  if (bad) { free(tok_seq); free(tok_j); return -1; }

#ifdef _OPENMP
  if (num_threads < 1) num_threads = 1;
#pragma omp parallel num_threads(num_threads)
#endif
  {
    double* x = (double*)malloc(sizeof(double) * (size_t)maxctx);
    double* qd = (double*)malloc(sizeof(double) * (size_t)head_dim);
    double* K = (double*)malloc(sizeof(double) * (size_t)maxctx * head_dim);
    double* V = (double*)malloc(sizeof(double) * (size_t)maxctx * head_dim);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t r = 0; r < total; ++r) {
      int64_t id = rows ? rows[r] : r;
      int64_t token = id / num_q_heads;
      int g = (int)(id % num_q_heads);
      int s = tok_seq[token];
      double* o = out + r * head_dim;
      int64_t n = chunk_lens ? chunk_lens[s] : 1;
      int64_t pos = (int64_t)context_lens[s] - n + tok_j[token];
      if (!seq_valid(block_table, context_lens, chunk_lens, s, page_size,
                     num_pages, max_pages_per_seq) || pos < 0) {
        for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
        continue;
      }
      const int h = g / group;
      attend_row(q + (token * num_q_heads + g) * (int64_t)head_dim, k_cache, v_cache, fmt,
                 fmt == KV_E4M3 ? (double)k_scale[h] : 1.0,
                 fmt == KV_E4M3 ? (double)v_scale[h] : 1.0,
                 block_table + (int64_t)s * max_pages_per_seq, pos, h, num_kv_heads,
                 head_dim, page_size, scale, o, qd, K, V, x);
    }
    free(x);
    free(qd);
    free(K);
    free(V);
  }
  free(tok_seq);
  free(tok_j);
  return 0;
}

int oracle_attention(const uint16_t* q, const uint16_t* k_cache,
                     const uint16_t* v_cache, const int32_t* block_table,
                     const int32_t* context_lens, const int32_t* chunk_lens,
                     int num_seqs, int num_q_heads, int num_kv_heads,
                     int head_dim, int page_size, int num_pages,
                     int max_pages_per_seq, double scale, const int64_t* rows,
                     int64_t nrows, double* out, int num_threads) {
  return attention_impl(q, k_cache, v_cache, KV_BF16, NULL, NULL, block_table, context_lens,
                        chunk_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, page_size,
                        num_pages, max_pages_per_seq, scale, rows, nrows, out, num_threads);
}

/* The same attention over an FP8 cache: K_t = e4m3(k) * k_scale[h], V_t =
 * e4m3(v) * v_scale[h], exactly, in double precision. */
int oracle_attention_fp8(const uint16_t* q, const uint8_t* k_cache, const uint8_t* v_cache,
                         const float* k_scale, const float* v_scale,
                         const int32_t* block_table, const int32_t* context_lens,
                         const int32_t* chunk_lens, int num_seqs, int num_q_heads,
                         int num_kv_heads, int head_dim, int page_size, int num_pages,
                         int max_pages_per_seq, double scale, const int64_t* rows,
                         int64_t nrows, double* out, int num_threads) {
  return attention_impl(q, k_cache, v_cache, KV_E4M3, k_scale, v_scale, block_table,
                        context_lens, chunk_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                        page_size, num_pages, max_pages_per_seq, scale, rows, nrows, out,
                        num_threads);
}

/*
 * Log-sum-exp merge of S partial attention states for each of R rows:
 * part_o [R, S, D] (each state normalised by its own softmax sum),
 * part_lse [R, S] natural-log sum of exp(scores) of that state's keys.
 * out = sum_i exp(lse_i - LSE) o_i with LSE = log sum_i exp(lse_i).  States
 * with lse = -inf hold no keys and are skipped; a row with none is zero.
 */
void oracle_combine(const double* part_o, const double* part_lse, int64_t R,
                    int S, int head_dim, double* out) {
  for (int64_t r = 0; r < R; ++r) {
    const double* lse = part_lse + r * S;
    double M = -INFINITY;
    for (int i = 0; i < S; ++i) if (lse[i] > M) M = lse[i];
    double* o = out + r * head_dim;
    for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
    if (M == -INFINITY) continue;
    double L = 0.0;
    for (int i = 0; i < S; ++i) if (lse[i] != -INFINITY) L += exp(lse[i] - M);
    for (int i = 0; i < S; ++i) {
      if (lse[i] == -INFINITY) continue;
      double w = exp(lse[i] - M) / L;
      for (int d = 0; d < head_dim; ++d) o[d] += w * part_o[(r * S + i) * head_dim + d];
    }
  }
}

/* OpenMP threads the library would use for num_threads <= 0 requests. */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------
 * Decode / prefill prologue: Q/K norm -> RoPE -> KV cache write.
 *
 * "Qwen 3" (TensorSharp model doc), section 3 "Forward graph": after the
 * fused QKV projection, per-head RMSNorm(Q) with attn_q_norm.weight and
 * per-head RMSNorm(K) with attn_k_norm.weight, then RoPE_NeoX(Q, K) at the
 * tokens' positions, then Q <- Q * (1/sqrt(headDim)), then (K, V) appended to
 * the KV cache.  Section 4.1: QK-norm is an RMSNorm over each head's headDim
 * values with a weight vector of size headDim; RoPE is NeoX-style with
 * frequencies from rope.freq_base and rope.scale (section 5: "frequency scale
 * divisor").  Section 4.3: epsilon from the config (typically 1e-6).
 * "Qwen3-14B" (pypto-lib), "Model structure, top down": decode_fwd runs
 * "Q/K norm -> RoPE" before the KV cache write; "Deployment configuration":
 * FP32 RMSNorm weights.
 *
 * Readings where the pages are silent:
 *  - RMSNorm(x) = x / sqrt(mean(x^2) + eps) * w, over the head's D values;
 *  - NeoX RoPE rotates the pair (x[i], x[i + D/2]), i < D/2, by the angle
 *    pos * f_i with f_i = base^(-2i/D) / scale:
 *      x'[i]       = x[i] cos - x[i + D/2] sin,
 *      x'[i + D/2] = x[i + D/2] cos + x[i] sin;
 *  - the input is the fused projection output, one row per token laid out as
 *    [Hq heads | Hkv heads (K) | Hkv heads (V)] of D values each;
 *  - the position of new token j of sequence s is ctx[s] - n[s] + j, as in
 *    the KV write; Q is multiplied by q_scale (1/sqrt(D) for the pages'
 *    folding, or 1 when the attention call applies the scale itself);
 *  - K is rounded to bf16 (round to nearest even, through float) before it
 *    is stored; V is stored bit for bit.
 * ------------------------------------------------------------------------ */

/* float -> bf16 bits, round to nearest even (finite inputs). */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  uint32_t rounding = 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)((u + rounding) >> 16);
}

/* RMSNorm of one head (section 4.1 QK-norm, section 4.3 epsilon). */
static void rms_norm_head(const double* x, const float* w, int d, double eps, double* y) {
  double ss = 0.0;
  for (int i = 0; i < d; ++i) ss += x[i] * x[i];
  double r = 1.0 / sqrt(ss / d + eps);
  for (int i = 0; i < d; ++i) y[i] = x[i] * r * (double)w[i];
}

/* NeoX rotary embedding of one head at position pos (section 4.1 RoPE). */
void oracle_rope_neox(double* y, int d, double pos, double base, double scale) {
  int half = d / 2;
  for (int i = 0; i < half; ++i) {
    double f = pow(base, -2.0 * i / d) / scale;
    double a = pos * f;
    double c = cos(a), s = sin(a);
    double x0 = y[i], x1 = y[i + half];
    y[i] = x0 * c - x1 * s;
    y[i + half] = x1 * c + x0 * s;
  }
}

/*
 * qkv      bf16 [num_tokens, (Hq + 2 Hkv) * D]
 * q_out    double [num_tokens, Hq, D] (normed, rotated, times q_scale); rows of
 *          invalid sequences are zero
 * k_cache, v_cache  bf16 pools, written like oracle_kv_write (K normed+rotated,
 *          rounded to bf16; V copied)
 * Returns the number of sequences skipped as invalid.
 */
int oracle_qk_norm_rope_write(const uint16_t* qkv, const float* wq, const float* wk,
                              double eps, double rope_base, double rope_scale,
                              double q_scale, double* q_out, uint16_t* k_cache,
                              uint16_t* v_cache, const int32_t* block_table,
                              const int32_t* context_lens, const int32_t* chunk_lens,
                              int64_t num_tokens, int num_seqs, int hq, int hkv, int d,
                              int page_size, int num_pages, int max_pages_per_seq) {
  const int64_t row_in = (int64_t)(hq + 2 * hkv) * d;
  const int64_t row_kv = (int64_t)hkv * d;
  double* x = (double*)malloc(sizeof(double) * d);
  double* y = (double*)malloc(sizeof(double) * d);
  int64_t token = 0;
  int skipped = 0;
  for (int s = 0; s < num_seqs; ++s) {
    int64_t n = chunk_lens ? chunk_lens[s] : 1;
    int ok = seq_valid(block_table, context_lens, chunk_lens, s, page_size, num_pages,
                       max_pages_per_seq);
    if (!ok) ++skipped;
    int64_t ctx = context_lens[s];
    for (int64_t j = 0; j < n && token < num_tokens; ++j, ++token) {
      const uint16_t* r = qkv + token * row_in;
      int64_t pos = ctx - n + j;
      for (int h = 0; h < hq; ++h) {
        double* dst = q_out + (token * hq + h) * d;
        if (!ok) {
          for (int i = 0; i < d; ++i) dst[i] = 0.0;
          continue;
        }
        for (int i = 0; i < d; ++i) x[i] = bf16_to_f64(r[h * d + i]);
        rms_norm_head(x, wq, d, eps, y);
        oracle_rope_neox(y, d, (double)pos, rope_base, rope_scale);
        for (int i = 0; i < d; ++i) dst[i] = y[i] * q_scale;
      }
      if (!ok) continue;
      int64_t page = block_table[(int64_t)s * max_pages_per_seq + pos / page_size];
      int64_t slot = page * page_size + pos % page_size;
      for (int h = 0; h < hkv; ++h) {
        for (int i = 0; i < d; ++i) x[i] = bf16_to_f64(r[(hq + h) * d + i]);
        rms_norm_head(x, wk, d, eps, y);
        oracle_rope_neox(y, d, (double)pos, rope_base, rope_scale);
        for (int i = 0; i < d; ++i)
          k_cache[slot * row_kv + h * d + i] = f32_to_bf16_rne((float)y[i]);
      }
      memcpy(v_cache + slot * row_kv, r + (int64_t)(hq + hkv) * d, (size_t)row_kv * 2);
    }
  }
  free(x);
  free(y);
  return skipped;
}

/* ------------------------------------------------------------------------
 * Exact top-k over rows of logits.
 *
 * pypto-serving PR #77 (page 3), "Exactness Design": an exact Top-32 of a
 * row's full-vocabulary logits (151936 real entries for Qwen3-14B), checked
 * against torch.topk(logits[:, :REAL_VOCAB], 32); the selector returns the
 * candidate values and token IDs.  The oracle is the plain definition: sort the
 * row's (value, index) pairs and take the first k.
 *
 * Readings where the pages are silent:
 *  - order: larger value first; NaN ranks above +inf (as torch.topk does);
 *    among equal values the smaller index comes first (the page fixes no tie
 *    order; this one is total, so the result is unique);
 *  - output: k values (as given) and their int32 indices, in that order.
 * ------------------------------------------------------------------------ */
typedef struct {
  float v;
  int32_t i;
} vi_pair;

static int nan_or(float x) { return x != x; }

/* qsort comparator: descending value (NaN largest), then ascending index. */
static int cmp_desc(const void* a, const void* b) {
  const vi_pair* x = (const vi_pair*)a;
  const vi_pair* y = (const vi_pair*)b;
  int xn = nan_or(x->v), yn = nan_or(y->v);
  if (xn != yn) return xn ? -1 : 1;
  if (!xn && x->v != y->v) return x->v > y->v ? -1 : 1;
  return (x->i < y->i) ? -1 : (x->i > y->i);
}

void oracle_topk(const float* logits, int64_t row_stride, int rows, int vocab, int k,
                 float* out_values, int32_t* out_indices) {
  vi_pair* buf = (vi_pair*)malloc(sizeof(vi_pair) * (size_t)(vocab > 0 ? vocab : 1));
  for (int r = 0; r < rows; ++r) {
    const float* row = logits + (int64_t)r * row_stride;
    for (int i = 0; i < vocab; ++i) {
      buf[i].v = row[i];
      buf[i].i = i;
    }
    qsort(buf, (size_t)vocab, sizeof(vi_pair), cmp_desc);
    for (int j = 0; j < k; ++j) {
      out_values[(int64_t)r * k + j] = buf[j].v;
      out_indices[(int64_t)r * k + j] = buf[j].i;
    }
  }
  free(buf);
}
