/*
 * spec_oracle.c -- CPU float64 oracle for the target-verify step of
 * speculative decoding.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: it exists so that tests, the smoke check and the CPU
 * baseline of the benchmark can compare the CUDA kernels against a plain,
 * slow, obviously correct definition.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it computes (the pages' definitions, written out):
 *
 *  1. Verify attention.  A request's verify block holds q_len known tokens
 *     [boundary, d1 .. dk] whose K/V already sit at the end of the request's
 *     paged KV cache.  Block row i attends causally to every cached key up to
 *     and including its own position, i.e. to the first
 *         L_i = seq_len - q_len + i + 1
 *     keys ("MTP and DFlash2 at long context on XPU", Part II "Why the target
 *     output stayed the same" and Part III "Reducing an eight-query verify
 *     with a severe shape cliff": each position gets its own cache length;
 *     "DFlash to dLLM self-spec, part 1", section 1.1, table of known inputs
 *     per verify row).  Query head h reads KV head h / (Hq/Hkv) (contiguous
 *     GQA groups).  Scores s_t = scale * <q, k_t>, softmax over t < L_i, and
 *     out = sum_t softmax_t * v_t.  The oracle uses the two-pass form:
 *     m = max_t s_t, w_t = exp(s_t - m), out = sum w_t v_t / sum w_t.
 *     No online softmax, no splits, no blocking.
 *
 *  2. Split merge ("Qwen3.8-27B-FP8" page, "Implemented execution path":
 *     split-context decode keeps compact online-softmax partials that a
 *     merge step combines).  A part s carries (o_s, lse_s) with
 *     lse_s = ln sum_{t in part} e^{s_t} and o_s the part's normalised
 *     output; the merge is lse = ln sum_s e^{lse_s},
 *     out = sum_s e^{lse_s - lse} o_s.
 *
 *  3. FP8 KV ("Qwen3.8-27B-FP8" page, "Implemented execution path": FP8 E4M3
 *     cache with per-token / per-KV-head FP16 scales over 64-channel
 *     blocks): element c of a cached K or V row is
 *         e4m3(byte_c) * fp16(scale[c / 64]).
 *     E4M3 is decoded from the OCP 8-bit floating point definition (bias 7,
 *     subnormals m * 2^-9, S.1111.111 is NaN, no infinities); FP16 and BF16
 *     from the IEEE binary16 / upper-half-of-binary32 definitions.
 *
 *  4. Greedy acceptance ("MTP and DFlash2 at long context on XPU", Part II:
 *     the runtime commits the accepted drafts and the target's token at the
 *     first disagreement; "DFlash to dLLM self-spec, part 1", section 1.1
 *     table and glossary "bonus token", section 1.6.1 commit_lens =
 *     accept_len + 1).  t_r = argmax over the fp32 logits of row r, lowest
 *     index on ties, NaN greater than every number (first NaN wins), -0 ==
 *     +0.  accept a = number of leading j = 1..k with draft[j] == t[j-1];
 *     next = t[a].
 *
 *  5. Per-request verify width ("Qwen3.8-27B-FP8" page: adaptive MTP K and
 *     the EWMA-driven DFlash2 verify width; "DFlash to dLLM self-spec,
 *     part 1", section 1.7.2: the verify length becomes a per-request
 *     scheduling decision).  Request b verifies q_b <= q_max rows in a block
 *     padded to q_max; block row i < q_b is token seq_len - q_b + i, rows
 *     i >= q_b do not exist (zero output, nothing appended or compared).
 *
 *  6. Commit and next-block preparation ("DFlash to dLLM self-spec,
 *     part 1", section 1.3.3: one kernel computes accept, bonus and the new
 *     sequence lengths, another the next block's ids, positions and cache
 *     locations; section 1.3.2: the GPU-side lengths advance without a copy
 *     to the host).  After accepting a drafts the cache holds the prefix,
 *     the boundary and d1..da: new_seq_len = seq_len - q_b + a + 1.  The
 *     bonus token opens the next block at position new_seq_len.
 *
 *  7. Stochastic verify ("MTP and DFlash2 at long context on XPU", Part II:
 *     sampling needs rejection sampling against target and draft
 *     probabilities; the rule is the speculative sampling of Leviathan et
 *     al. 2023, "Fast Inference from Transformers via Speculative Decoding",
 *     and Chen et al. 2023).  p_j = softmax(logits[b, j] / T_b) is the
 *     target's distribution for the token after block position j; q_j is
 *     the drafter's distribution that proposed d_j (one-hot at d_j for a
 *     greedy drafter).  Draft j is accepted iff u_j * q_j(d_j) <
 *     p_{j-1}(d_j); at the first rejection the next token is drawn from the
 *     normalised residual max(0, p_{j-1} - q_j); when every draft is
 *     accepted it is drawn from p_{q_b-1}.  A draw from weights w with the
 *     uniform u is the smallest v whose running sum exceeds u * sum(w).
 *
 *  8. DFlash2 candidate selector ("MTP and DFlash2 at long context on XPU",
 *     "The part that makes DFlash2 different" and "Selector and recurrent
 *     math"; "Qwen3.8-27B-FP8" page: selector_rank = 256, selector_top_k =
 *     16, and an exact MAP over the chain as an option).  Each draft
 *     position t = 1 .. P-1 keeps the K best tokens of its candidate logits
 *     (larger logit first, lower token id on ties).  A transition from
 *     candidate a at t-1 (the boundary token at t = 0) to candidate b at t
 *     scores S_t(a, b) = U_t(b) + sum_r A[a, r] H_t[r] B[b, r], with U_t(b)
 *     the candidate's logit, A and B the predecessor and successor
 *     codebooks (rows indexed by token id, rank R) and H_t = W_H h_t the
 *     projection of the draft hidden state at t.  The greedy walk starts at
 *     the boundary and takes at each position the best successor of the
 *     token already chosen (lowest candidate rank on ties); the MAP walk
 *     maximises the sum of S_t along the chain.
 *
 * Parity of this oracle against any engine on the pages is unpinned: the
 * pages print no output for a concrete input tensor.  It is pinned instead
 * by tests against library routines (torch scaled-dot-product attention in
 * float64, torch's float8_e4m3fn and numpy's float16 decoders, numpy
 * argmax), closed forms, invariants and the pages' worked accept examples.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_PAGE (-2)
#define ORACLE_ERR_NOMEM (-3)

/* ---- exact decoders, written from the format definitions ---------------- */

double oracle_bf16_to_double(uint16_t h) {
  /* bfloat16 is the upper half of an IEEE binary32 */
  uint32_t bits = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

double oracle_fp16_to_double(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 0x1F, m = h & 0x3FF;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24); /* subnormal: m * 2^-14 * 2^-10 */
  } else if (e == 31) {
    v = m ? NAN : INFINITY;
  } else {
    v = ldexp(1.0 + (double)m / 1024.0, e - 15);
  }
  return s ? -v : v;
}

double oracle_e4m3_to_double(uint8_t b) {
  int s = (b >> 7) & 1, e = (b >> 3) & 0xF, m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN; /* S.1111.111: the only NaN, no inf */
  if (e == 0) {
    v = ldexp((double)m, -9); /* subnormal: m/8 * 2^(1-7) */
  } else {
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  }
  return s ? -v : v;
}

void oracle_decode_bf16(const uint16_t* x, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_double(x[i]);
}
void oracle_decode_fp16(const uint16_t* x, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_fp16_to_double(x[i]);
}
void oracle_decode_e4m3(const uint8_t* x, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_to_double(x[i]);
}

/* ---- verify attention ------------------------------------------------------ */

typedef struct {
  int32_t batch, q_len, hq, hkv, d, page_size, num_pages, max_pages, kv_fp8;
  const uint16_t* q;       /* bf16 bits [batch, q_len, hq, d] */
  const void* k_pages;     /* bf16 bits or e4m3 bytes [num_pages, hkv, page_size, d] */
  const void* v_pages;
  const uint16_t* k_scales; /* fp16 bits [num_pages, hkv, page_size, d/64] (fp8 only) */
  const uint16_t* v_scales;
  const int32_t* page_table; /* [batch, max_pages] */
  const int32_t* seq_lens;   /* [batch], block included */
  const int32_t* q_lens;     /* [batch] rows per request, or NULL: q_len */
} oracle_attn_problem;

/* Rows of request b's block: q_lens[b] clamped to [0, q_max], or q_max. */
static int32_t block_rows(const int32_t* q_lens, int b, int32_t q_max) {
  if (!q_lens) return q_max;
  int32_t v = q_lens[b];
  return v < 0 ? 0 : (v > q_max ? q_max : v);
}

/* Element c of the cached K (or V) row of token t of request b, KV head g.
 * Returns 0 and writes the row, or ORACLE_ERR_PAGE for a page id outside the
 * pool. */
static int load_kv_row(const oracle_attn_problem* p, int is_v, int b, int g,
                       int64_t t, double* row) {
  const int ps = p->page_size, d = p->d;
  int64_t page_slot = t / ps;
  if (page_slot >= p->max_pages) return ORACLE_ERR_PAGE;
  int32_t page = p->page_table[(int64_t)b * p->max_pages + page_slot];
  if (page < 0 || page >= p->num_pages) return ORACLE_ERR_PAGE;
  int64_t slot = t % ps;
  int64_t base = (((int64_t)page * p->hkv + g) * ps + slot) * d;
  if (!p->kv_fp8) {
    const uint16_t* src = (const uint16_t*)(is_v ? p->v_pages : p->k_pages);
    for (int c = 0; c < d; ++c) row[c] = oracle_bf16_to_double(src[base + c]);
  } else {
    const uint8_t* src = (const uint8_t*)(is_v ? p->v_pages : p->k_pages);
    const uint16_t* sc = is_v ? p->v_scales : p->k_scales;
    int64_t sbase = (((int64_t)page * p->hkv + g) * ps + slot) * (d / 64);
    for (int c = 0; c < d; ++c)
      row[c] = oracle_e4m3_to_double(src[base + c]) *
               oracle_fp16_to_double(sc[sbase + c / 64]);
  }
  return ORACLE_OK;
}

/* One output row: request b, block row i, query head h, keys restricted to
 * [key_begin, key_end) intersected with the causal window [0, L_i). */
static int attention_row(const oracle_attn_problem* p, int b, int i, int h,
                         int64_t key_begin, int64_t key_end, double scale,
                         double* s_buf, double* krow, double* out, double* lse) {
  const int d = p->d;
  const int group = p->hq / p->hkv;
  const int g = h / group;
  const int32_t qb = block_rows(p->q_lens, b, p->q_len);
  const int64_t causal = i < qb ? (int64_t)p->seq_lens[b] - qb + i + 1 : 0;
  int64_t lo = key_begin > 0 ? key_begin : 0;
  int64_t hi = causal;
  if (key_end >= 0 && key_end < hi) hi = key_end;
  for (int c = 0; c < d; ++c) out[c] = 0.0;
  if (hi <= lo) {
    *lse = -INFINITY;
    return ORACLE_OK;
  }
  double qrow[1024];
  const uint16_t* qsrc = p->q + (((int64_t)b * p->q_len + i) * p->hq + h) * d;
  for (int c = 0; c < d; ++c) qrow[c] = oracle_bf16_to_double(qsrc[c]);

  /* pass 1: all scores and their maximum */
  double m = -INFINITY;
  for (int64_t t = lo; t < hi; ++t) {
    int rc = load_kv_row(p, 0, b, g, t, krow);
    if (rc) return rc;
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += qrow[c] * krow[c];
    double s = scale * acc;
    s_buf[t - lo] = s;
    if (s > m) m = s;
  }
  /* pass 2: weights and the weighted sum of V rows */
  double den = 0.0;
  for (int64_t t = lo; t < hi; ++t) {
    double w = exp(s_buf[t - lo] - m);
    den += w;
    int rc = load_kv_row(p, 1, b, g, t, krow);
    if (rc) return rc;
    for (int c = 0; c < d; ++c) out[c] += w * krow[c];
  }
  for (int c = 0; c < d; ++c) out[c] /= den;
  *lse = m + log(den);
  return ORACLE_OK;
}

/*
 * Verify attention for a list of rows.
 *   rows:  flat row ids r = (b * q_len + i) * hq + h, or NULL for all
 *          batch * q_len * hq rows in that order.
 *   key_begin/key_end: restrict the keys to [key_begin, key_end) (key_end < 0
 *          means no upper limit) on top of the causal window; used to form
 *          split partials.
 *   out:   [n_rows, d] float64;  lse: [n_rows] (natural log) or NULL.
 * Returns 0, ORACLE_ERR_ARG for bad shapes, ORACLE_ERR_PAGE for a page id
 * outside the pool, ORACLE_ERR_NOMEM.
 */
int oracle_verify_attention(int32_t batch, int32_t q_len, int32_t hq,
                            int32_t hkv, int32_t d, int32_t page_size,
                            int32_t num_pages, int32_t max_pages,
                            int32_t kv_fp8, const uint16_t* q,
                            const void* k_pages, const void* v_pages,
                            const uint16_t* k_scales, const uint16_t* v_scales,
                            const int32_t* page_table, const int32_t* seq_lens,
                            const int32_t* q_lens, double scale,
                            const int64_t* rows, int64_t n_rows,
                            int64_t key_begin, int64_t key_end, double* out,
                            double* lse, int32_t nthreads) {
  if (batch < 0 || q_len < 1 || hq < 1 || hkv < 1 || hq % hkv || d < 1 ||
      d > 1024 || page_size < 1 || num_pages < 0 || max_pages < 0)
    return ORACLE_ERR_ARG;
  if (kv_fp8 && (d % 64 || !k_scales || !v_scales)) return ORACLE_ERR_ARG;
  oracle_attn_problem p = {batch,   q_len,     hq,       hkv,      d,
                           page_size, num_pages, max_pages, kv_fp8, q,
                           k_pages, v_pages,   k_scales, v_scales, page_table,
                           seq_lens, q_lens};
  const int64_t total = (int64_t)batch * q_len * hq;
  if (!rows) n_rows = total;
  int64_t max_len = 0;
  for (int b = 0; b < batch; ++b)
    if (seq_lens[b] > max_len) max_len = seq_lens[b];
  int err = ORACLE_OK;
#ifdef _OPENMP
  if (nthreads < 1) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
  {
    double* s_buf = (double*)malloc(sizeof(double) * (size_t)(max_len + 1));
    double* krow = (double*)malloc(sizeof(double) * (size_t)d);
    double dummy;
    if (!s_buf || !krow) {
#ifdef _OPENMP
#pragma omp critical
#endif
      err = ORACLE_ERR_NOMEM;
    } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
      for (int64_t n = 0; n < n_rows; ++n) {
        int64_t r = rows ? rows[n] : n;
        if (r < 0 || r >= total) {
#ifdef _OPENMP
#pragma omp critical
#endif
          err = ORACLE_ERR_ARG;
          continue;
        }
        int h = (int)(r % hq);
        int i = (int)((r / hq) % q_len);
        int b = (int)(r / ((int64_t)hq * q_len));
        int rc = attention_row(&p, b, i, h, key_begin, key_end, scale, s_buf,
                               krow, out + n * d, lse ? lse + n : &dummy);
        if (rc) {
#ifdef _OPENMP
#pragma omp critical
#endif
          err = rc;
        }
      }
    }
    free(s_buf);
    free(krow);
  }
  return err;
}

/*
 * Merge of split partials: lse = ln sum_s e^{lse_s},
 * out = sum_s e^{lse_s - lse} o_s.  o: [n_parts, d]; parts with
 * lse_s = -inf carry no weight; all parts empty gives out = 0, lse = -inf.
 */
void oracle_lse_merge(int32_t n_parts, int32_t d, const double* lse,
                      const double* o, double* out, double* lse_out) {
  double m = -INFINITY;
  for (int s = 0; s < n_parts; ++s)
    if (lse[s] > m) m = lse[s];
  for (int c = 0; c < d; ++c) out[c] = 0.0;
  if (m == -INFINITY) {
    *lse_out = -INFINITY;
    return;
  }
  double den = 0.0;
  for (int s = 0; s < n_parts; ++s) den += exp(lse[s] - m);
  double total = m + log(den);
  for (int s = 0; s < n_parts; ++s) {
    if (lse[s] == -INFINITY) continue;
    double w = exp(lse[s] - total);
    for (int c = 0; c < d; ++c) out[c] += w * o[(int64_t)s * d + c];
  }
  *lse_out = total;
}

/* ---- encoders and block KV append ---------------------------------------------
 *
 * Quantise-on-write of the FP8 cache ("Qwen3.8-27B-FP8" page, "Implemented
 * execution path": E4M3 with per-token / per-KV-head FP16 scales over
 * 64-channel blocks).  The pages fix the format, not the rounding rule;
 * the rule taken here (and stated in the C header of the library) is
 *   amax  = max |x| over the 64-channel block, x the bf16 input as float
 *   scale = fp16 round-to-nearest-even of (float)(amax / 448), computed as
 *           an IEEE single-precision division; 1 if that rounds to zero
 *   byte  = E4M3 round-to-nearest-even of (float)(x / scale), saturated to
 *           +-448.
 * Both encoders round an exactly known value once, from the definitions
 * of the formats: fp16 has 10 fraction bits, exponent bias 15, subnormal
 * quantum 2^-24; E4M3 has 3 fraction bits, bias 7, subnormal quantum 2^-9,
 * largest finite 448. */

uint16_t oracle_fp16_from_double(double x) {
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (isnan(x)) return 0x7E00;
  if (a == 0.0) return sign;
  double q;                 /* quantum at |x| */
  int e;
  frexp(a, &e);             /* a = m * 2^e, m in [0.5, 1) */
  if (e - 1 < -14) q = ldexp(1.0, -24);
  else q = ldexp(1.0, e - 1 - 10);
  double r = rint(a / q) * q;   /* round half to even (default mode) */
  if (r >= 65520.0 || isinf(a)) return sign | 0x7C00;  /* overflow: inf */
  if (r < ldexp(1.0, -14)) return sign | (uint16_t)(r / ldexp(1.0, -24));
  frexp(r, &e);
  int E = e - 1;
  uint16_t mant = (uint16_t)((r / ldexp(1.0, E) - 1.0) * 1024.0);
  return sign | (uint16_t)((E + 15) << 10) | mant;
}

uint8_t oracle_e4m3_from_double(double x) {
  uint8_t sign = signbit(x) ? 0x80 : 0;
  double a = fabs(x);
  if (isnan(x)) return 0x7F;
  if (a >= 448.0) return sign | 0x7E;          /* saturate (inf included) */
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);
  double q = (e - 1 < -6) ? ldexp(1.0, -9) : ldexp(1.0, e - 1 - 3);
  double r = rint(a / q) * q;
  if (r >= 448.0) return sign | 0x7E;
  if (r < ldexp(1.0, -6)) return sign | (uint8_t)(r / ldexp(1.0, -9));
  frexp(r, &e);
  int E = e - 1;
  uint8_t mant = (uint8_t)((r / ldexp(1.0, E) - 1.0) * 8.0);
  return sign | (uint8_t)((E + 7) << 3) | mant;
}

void oracle_encode_fp16(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_fp16_from_double(x[i]);
}
void oracle_encode_e4m3(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_from_double(x[i]);
}

/*
 * Block KV append.  Block row i < q_b of request b (q_b = q_lens[b], or
 * q_len when q_lens is NULL) is token t = seq_lens[b] - q_b + i; its K and V rows of KV head g go to page
 * page_table[b, t / page_size], slot t % page_size ("DFlash to dLLM
 * self-spec, part 1", section 1.3.2 "KV over-allocation" and section 1.3.3:
 * block ids, positions and cache loc prepared in one kernel).
 *   k_new, v_new: bf16 bits [B, q_len, hkv, d]
 *   pools / scales: updated in place (scales only when kv_fp8)
 *   positions [B, q_len]: t, or -1 when t < 0 or i >= q_b
 *   cache_loc [B, q_len]: page * page_size + slot, or -1 when the token has
 *   no slot (i >= q_b, t < 0, t beyond the table, page id outside the
 *   pool); such rows are not written.
 */
int oracle_kv_append(int32_t batch, int32_t q_len, int32_t hkv, int32_t d,
                     int32_t page_size, int32_t num_pages, int32_t max_pages,
                     int32_t kv_fp8, const uint16_t* k_new,
                     const uint16_t* v_new, void* k_pages, void* v_pages,
                     uint16_t* k_scales, uint16_t* v_scales,
                     const int32_t* page_table, const int32_t* seq_lens,
                     const int32_t* q_lens, int32_t* positions,
                     int64_t* cache_loc) {
  if (batch < 0 || q_len < 1 || hkv < 1 || d < 1 || page_size < 1 ||
      (kv_fp8 && d % 64))
    return ORACLE_ERR_ARG;
  const int64_t max_tokens = (int64_t)max_pages * page_size;
  for (int b = 0; b < batch; ++b) {
    const int32_t qb = block_rows(q_lens, b, q_len);
    for (int i = 0; i < q_len; ++i) {
      const int64_t t = (int64_t)seq_lens[b] - qb + i;
      int64_t loc = -1;
      int32_t page = -1;
      if (i >= qb) {
        positions[(int64_t)b * q_len + i] = -1;
        cache_loc[(int64_t)b * q_len + i] = -1;
        continue;
      }
      if (t >= 0 && t < max_tokens) {
        page = page_table[(int64_t)b * max_pages + t / page_size];
        if (page >= 0 && page < num_pages)
          loc = (int64_t)page * page_size + t % page_size;
      }
      positions[(int64_t)b * q_len + i] = t >= 0 ? (int32_t)t : -1;
      cache_loc[(int64_t)b * q_len + i] = loc;
      if (loc < 0) continue;
      for (int g = 0; g < hkv; ++g) {
        const int64_t row = ((int64_t)page * hkv + g) * page_size + t % page_size;
        const int64_t src = (((int64_t)b * q_len + i) * hkv + g) * d;
        for (int kv = 0; kv < 2; ++kv) {
          const uint16_t* in = kv ? v_new : k_new;
          if (!kv_fp8) {
            uint16_t* dst = (uint16_t*)(kv ? v_pages : k_pages);
            for (int c = 0; c < d; ++c) dst[row * d + c] = in[src + c];
            continue;
          }
          uint8_t* dst = (uint8_t*)(kv ? v_pages : k_pages);
          uint16_t* sc = kv ? v_scales : k_scales;
          for (int blk = 0; blk < d / 64; ++blk) {
            float amax = 0.0f;
            for (int c = 0; c < 64; ++c) {
              float x = (float)oracle_bf16_to_double(in[src + blk * 64 + c]);
              if (fabsf(x) > amax) amax = fabsf(x);
            }
            float q = amax / 448.0f;            /* IEEE single division */
            uint16_t sbits = oracle_fp16_from_double((double)q);
            if ((sbits & 0x7FFF) == 0) sbits = 0x3C00;   /* 1.0 */
            float s = (float)oracle_fp16_to_double(sbits);
            sc[row * (d / 64) + blk] = sbits;
            for (int c = 0; c < 64; ++c) {
              float x = (float)oracle_bf16_to_double(in[src + blk * 64 + c]);
              float y = x / s;                    /* IEEE single division */
              dst[row * d + blk * 64 + c] = oracle_e4m3_from_double((double)y);
            }
          }
        }
      }
    }
  }
  return ORACLE_OK;
}

/* ---- greedy acceptance ------------------------------------------------------ */

/* argmax with the lowest index on ties; NaN ranks above every number and
 * the first NaN wins; -0 and +0 compare equal. */
static int64_t row_argmax(const float* x, int64_t n) {
  int64_t best = 0;
  float bv = x[0];
  if (isnan(bv)) return 0;
  for (int64_t v = 1; v < n; ++v) {
    float xv = x[v];
    if (isnan(xv)) return v;
    if (xv > bv) {
      bv = xv;
      best = v;
    }
  }
  return best;
}

/*
 * logits: [batch * q_len, vocab] fp32, row (b, j) scores the token after
 *         block position j.
 * draft_ids: [batch, q_len]; column 0 is the boundary token (not compared),
 *         columns 1..q_len-1 are the drafts d1..dk.
 * q_lens: [batch] rows per request (NULL: q_len); only rows j < q_b and
 *         drafts 1..q_b-1 take part.  A request with q_b = 0 is idle:
 *         accept 0, next -1, nothing committed.
 * accept_len/next_token: [batch].  out_tokens [batch, q_len] (optional):
 *         d1..da, then next, then -1.  argmax_rows [batch * q_len] (optional).
 * seq_lens -> new_seq_lens (both optional, [batch]): seq_len - q_b + a + 1,
 *         the cache length once the boundary and d1..da are committed
 *         (seq_len for an idle request).
 */
int oracle_greedy_accept(const float* logits, const int32_t* draft_ids,
                         const int32_t* q_lens, int32_t batch, int32_t q_len,
                         int64_t vocab, const int32_t* seq_lens,
                         int32_t* new_seq_lens, int32_t* accept_len,
                         int32_t* next_token, int32_t* out_tokens,
                         int32_t* argmax_rows, int32_t nthreads) {
  if (batch < 0 || q_len < 1 || vocab < 1) return ORACLE_ERR_ARG;
  const int64_t rows = (int64_t)batch * q_len;
  int32_t* t = (int32_t*)malloc(sizeof(int32_t) * (size_t)(rows ? rows : 1));
  if (!t) return ORACLE_ERR_NOMEM;
#ifdef _OPENMP
  if (nthreads < 1) nthreads = omp_get_max_threads();
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
#endif
  for (int64_t r = 0; r < rows; ++r)
    t[r] = (int32_t)row_argmax(logits + r * vocab, vocab);
  for (int b = 0; b < batch; ++b) {
    const int32_t* dr = draft_ids + (int64_t)b * q_len;
    const int32_t* tb = t + (int64_t)b * q_len;
    const int32_t qb = block_rows(q_lens, b, q_len);
    int32_t* ot = out_tokens ? out_tokens + (int64_t)b * q_len : NULL;
    if (ot)
      for (int j = 0; j < q_len; ++j) ot[j] = -1;
    if (qb == 0) {
      accept_len[b] = 0;
      next_token[b] = -1;
      if (new_seq_lens) new_seq_lens[b] = seq_lens[b];
      continue;
    }
    int a = 0;
    while (a + 1 < qb && dr[a + 1] == tb[a]) ++a;
    accept_len[b] = a;
    next_token[b] = tb[a];
    if (ot) {
      for (int j = 0; j < a; ++j) ot[j] = dr[j + 1];
      ot[a] = tb[a];
    }
    if (new_seq_lens) new_seq_lens[b] = seq_lens[b] - qb + a + 1;
  }
  if (argmax_rows) memcpy(argmax_rows, t, sizeof(int32_t) * (size_t)rows);
  free(t);
  return ORACLE_OK;
}

/* ---- verify width policy and next-block preparation ------------------------ */

#define ORACLE_WIDTH_FIXED 0
#define ORACLE_WIDTH_EWMA 1
#define ORACLE_WIDTH_DOUBLING 2

/*
 * After a verify step: choose each request's next width and lay out its next
 * block.  For request b with q_b rows this step and a accepted drafts:
 *
 *   FIXED:    w = q_max.
 *   EWMA      ("Qwen3.8-27B-FP8" page, DFlash2 adaptive width: an EWMA of
 *             the accepted count, verify ewma + 1.5 rows, floor of two):
 *             e <- (1 - alpha) * e + alpha * a, each operation rounded to
 *             float32, no fused multiply-add; w = ceil(e + offset) clamped
 *             to [min_width, q_max].  state[b] holds e.
 *   DOUBLING  ("Qwen3.8-27B-FP8" page, adaptive MTP K: start at K = 1,
 *             double after full acceptance, back off after rejection):
 *             K <- 2K if a == q_b - 1 else K / 2 (integer halving), clamped
 *             to [1, max(1, q_max - 1)]; w = min(K + 1, q_max).  state[b]
 *             holds K.
 *
 * An idle request (q_b = 0) keeps its state and stays idle (w = 0).
 * The next block of an active request starts at p = new_seq_lens[b]:
 *   next_q_lens[b] = w, next_seq_lens[b] = p + w,
 *   block_ids[b, :] = [next_token, mask_id x (w - 1), -1 ...],
 *   positions[b, i] = p + i (i < w, else -1),
 *   cache_loc[b, i] = page_table[b, (p+i)/ps] * ps + (p+i) % ps, or -1 when
 *   i >= w or the slot is not reserved (past the table, page id outside the
 *   pool).  Returns the number of rows i < w without a reserved slot.
 */
int64_t oracle_prepare_next_block(
    int32_t policy, int32_t q_max, int32_t min_width, float alpha,
    float offset, int32_t batch, const int32_t* q_lens,
    const int32_t* accept_len, const int32_t* next_token,
    const int32_t* new_seq_lens, float* state, int32_t mask_id,
    const int32_t* page_table, int32_t max_pages, int32_t page_size,
    int32_t num_pages, int32_t* next_q_lens, int32_t* next_seq_lens,
    int32_t* block_ids, int32_t* positions, int64_t* cache_loc) {
  if (batch < 0 || q_max < 1 || page_size < 1 || policy < 0 || policy > 2)
    return ORACLE_ERR_ARG;
  int64_t missing = 0;
  for (int b = 0; b < batch; ++b) {
    const int32_t qb = block_rows(q_lens, b, q_max);
    const int32_t a = accept_len[b];
    int32_t w = 0;
    if (qb > 0) {
      if (policy == ORACLE_WIDTH_FIXED) {
        w = q_max;
      } else if (policy == ORACLE_WIDTH_EWMA) {
        const float keep = 1.0f - alpha;
        const float old_part = keep * state[b];
        const float new_part = alpha * (float)a;
        const float e = old_part + new_part;
        state[b] = e;
        const float wf = ceilf(e + offset);
        if (!(wf < (float)q_max)) w = q_max;   /* also NaN */
        else if (wf < (float)min_width) w = min_width;
        else w = (int32_t)wf;
        if (w > q_max) w = q_max;
        if (w < 1) w = 1;
      } else {
        const int32_t kmax = q_max - 1 > 1 ? q_max - 1 : 1;
        int32_t k = (int32_t)state[b];
        k = a == qb - 1 ? 2 * k : k / 2;
        if (k < 1) k = 1;
        if (k > kmax) k = kmax;
        state[b] = (float)k;
        w = k + 1 < q_max ? k + 1 : q_max;
      }
    }
    const int64_t pos0 = new_seq_lens[b];
    next_q_lens[b] = w;
    next_seq_lens[b] = (int32_t)(pos0 + w);
    for (int i = 0; i < q_max; ++i) {
      const int64_t o = (int64_t)b * q_max + i;
      if (i >= w) {
        block_ids[o] = -1;
        positions[o] = -1;
        cache_loc[o] = -1;
        continue;
      }
      const int64_t t = pos0 + i;
      block_ids[o] = i == 0 ? next_token[b] : mask_id;
      positions[o] = (int32_t)t;
      int64_t loc = -1;
      if (t >= 0 && t / page_size < max_pages) {
        const int32_t page = page_table[(int64_t)b * max_pages + t / page_size];
        if (page >= 0 && page < num_pages)
          loc = (int64_t)page * page_size + t % page_size;
      }
      cache_loc[o] = loc;
      if (loc < 0) ++missing;
    }
  }
  return missing;
}

/* ---- stochastic verify (rejection sampling) ------------------------------- */

/* Row softmax statistics at temperature t: m = max_v x_v, z = sum_v
 * exp((x_v - m) / t).  p(v) = exp((x_v - m) / t) / z. */
static void softmax_stats(const float* x, int64_t n, double t, double* m,
                          double* z) {
  double mx = -INFINITY;
  for (int64_t v = 0; v < n; ++v)
    if ((double)x[v] > mx) mx = (double)x[v];
  double s = 0.0;
  for (int64_t v = 0; v < n; ++v) s += exp(((double)x[v] - mx) / t);
  *m = mx;
  *z = s;
}

/*
 * logits       fp32 [batch * q_len, vocab]
 * draft_ids    int32 [batch, q_len] (column 0 the boundary token)
 * draft_probs  fp32 [batch, q_len - 1, vocab]: row j-1 is q_j, the
 *              distribution draft j was drawn from; NULL for greedy drafts
 * q_lens       optional [batch] rows per request (as greedy accept)
 * temperature  fp32 [batch], > 0
 * u_accept     fp32 [batch, q_len - 1] uniforms in [0, 1) for the accept
 *              tests; u_sample fp32 [batch] the uniform of the final draw
 * seq_lens / new_seq_lens, accept_len, next_token, out_tokens: as greedy
 * margin        optional fp64 [batch] out: the smallest distance of any
 *              decision this request took from its threshold, relative to
 *              the quantities compared (|u q - p| / max(p, q) for a test;
 *              distance of u * W from the chosen interval's ends / W for
 *              the draw).  A request with a small margin may legitimately
 *              come out differently under another rounding.
 */
int oracle_stochastic_accept(const float* logits, const int32_t* draft_ids,
                             const float* draft_probs, const int32_t* q_lens,
                             int32_t batch, int32_t q_len, int64_t vocab,
                             const float* temperature, const float* u_accept,
                             const float* u_sample, const int32_t* seq_lens,
                             int32_t* new_seq_lens, int32_t* accept_len,
                             int32_t* next_token, int32_t* out_tokens,
                             double* margin, int32_t nthreads) {
  if (batch < 0 || q_len < 1 || vocab < 1) return ORACLE_ERR_ARG;
  int err = ORACLE_OK;
#ifdef _OPENMP
  if (nthreads < 1) nthreads = omp_get_max_threads();
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
#endif
  for (int b = 0; b < batch; ++b) {
    const int32_t qb = block_rows(q_lens, b, q_len);
    const int32_t* dr = draft_ids + (int64_t)b * q_len;
    int32_t* ot = out_tokens ? out_tokens + (int64_t)b * q_len : NULL;
    if (ot)
      for (int j = 0; j < q_len; ++j) ot[j] = -1;
    double mg = INFINITY;
    if (qb == 0) {
      accept_len[b] = 0;
      next_token[b] = -1;
      if (new_seq_lens) new_seq_lens[b] = seq_lens[b];
      if (margin) margin[b] = mg;
      continue;
    }
    const double t = (double)temperature[b];
    if (!(t > 0.0)) {
#ifdef _OPENMP
#pragma omp critical
#endif
      err = ORACLE_ERR_ARG;
      continue;
    }
    int a = 0;
    int rejected = 0;
    double m = 0.0, z = 0.0;
    for (int j = 1; j < qb; ++j) {
      const float* row = logits + ((int64_t)b * q_len + j - 1) * vocab;
      softmax_stats(row, vocab, t, &m, &z);
      const int32_t d = dr[j];
      const double p = (d >= 0 && d < vocab)
                           ? exp(((double)row[d] - m) / t) / z : 0.0;
      double q = 1.0;
      if (draft_probs && d >= 0 && d < vocab)
        q = (double)draft_probs[((int64_t)b * (q_len - 1) + j - 1) * vocab + d];
      const double u = (double)u_accept[(int64_t)b * (q_len - 1) + j - 1];
      const double scale = p > q ? p : q;
      if (scale > 0.0) {
        const double dist = fabs(u * q - p) / scale;
        if (dist < mg) mg = dist;
      }
      if (u * q < p) {
        ++a;
      } else {
        rejected = 1;
        break;
      }
    }
    /* the final draw: from row a, minus q_{a+1} after a rejection */
    const float* row = logits + ((int64_t)b * q_len + a) * vocab;
    softmax_stats(row, vocab, t, &m, &z);
    const float* qrow = NULL;
    if (rejected && draft_probs)
      qrow = draft_probs + ((int64_t)b * (q_len - 1) + a) * vocab;
    const int32_t drej = rejected ? dr[a + 1] : -1;
    double total = 0.0;
    for (int64_t v = 0; v < vocab; ++v) {
      double w = exp(((double)row[v] - m) / t) / z;
      if (rejected) {
        const double qv = qrow ? (double)qrow[v] : (v == drej ? 1.0 : 0.0);
        w = w > qv ? w - qv : 0.0;
      }
      total += w;
    }
    int use_residual = rejected && total > 0.0;
    if (rejected && !use_residual) { /* p == q: fall back to p itself */
      total = 0.0;
      for (int64_t v = 0; v < vocab; ++v) total += exp(((double)row[v] - m) / t) / z;
    }
    const double target = (double)u_sample[b] * total;
    double cum = 0.0, prev = 0.0;
    int64_t pick = -1;
    for (int64_t v = 0; v < vocab; ++v) {
      double w = exp(((double)row[v] - m) / t) / z;
      if (use_residual) {
        const double qv = qrow ? (double)qrow[v] : (v == drej ? 1.0 : 0.0);
        w = w > qv ? w - qv : 0.0;
      }
      prev = cum;
      cum += w;
      if (cum > target) {
        pick = v;
        break;
      }
    }
    if (pick < 0) { /* rounding left u * W at the very end: last nonzero */
      for (int64_t v = vocab - 1; v >= 0; --v) {
        double w = exp(((double)row[v] - m) / t) / z;
        if (use_residual) {
          const double qv = qrow ? (double)qrow[v] : (v == drej ? 1.0 : 0.0);
          w = w > qv ? w - qv : 0.0;
        }
        if (w > 0.0) {
          pick = v;
          break;
        }
      }
      prev = cum = target;
    }
    if (total > 0.0) {
      const double lo = (target - prev) / total, hi = (cum - target) / total;
      const double dist = lo < hi ? lo : hi;
      if (dist < mg) mg = dist;
    }
    accept_len[b] = a;
    next_token[b] = (int32_t)pick;
    if (ot) {
      for (int j = 0; j < a; ++j) ot[j] = dr[j + 1];
      ot[a] = (int32_t)pick;
    }
    if (new_seq_lens) new_seq_lens[b] = seq_lens[b] - qb + a + 1;
    if (margin) margin[b] = mg;
  }
  return err;
}

/* ---- DFlash2 candidate selector -------------------------------------------- */

#define ORACLE_SELECT_GREEDY 0
#define ORACLE_SELECT_MAP 1

/* The k best entries of x[0..n) in order: larger value first, lower index on
 * ties.  Insertion into a sorted list of k. */
static void top_k(const float* x, int64_t n, int k, int32_t* ids, float* vals) {
  int have = 0;
  for (int64_t v = 0; v < n; ++v) {
    const float xv = x[v];
    if (have == k && !(xv > vals[k - 1])) continue; /* ties keep the lower id */
    int pos = have < k ? have : k - 1;
    while (pos > 0 && xv > vals[pos - 1]) {
      vals[pos] = vals[pos - 1];
      ids[pos] = ids[pos - 1];
      --pos;
    }
    vals[pos] = xv;
    ids[pos] = (int32_t)v;
    if (have < k) ++have;
  }
  for (int i = have; i < k; ++i) {
    ids[i] = -1;
    vals[i] = -INFINITY;
  }
}

/*
 * cand_logits  fp32 [B, P-1, V]: row t-1 scores draft position t
 * boundary     int32 [B]: the verified token at position 0
 * hidden       bf16 bits [B, P-1, D]: draft hidden state of position t
 * w_h          bf16 bits [R, D]: the projection H = W_H h
 * code_a, code_b  bf16 bits [V, R]: predecessor / successor codebooks
 * mode         ORACLE_SELECT_GREEDY or ORACLE_SELECT_MAP
 * cand_ids     int32 [B, P-1, K] out; cand_logit fp32-as-double [B, P-1, K]
 * trans        fp64 [B, P-1, K, K] out: trans[b, t-1, a, c] = S_t(a, c)
 *              with a the predecessor's rank (t = 1: only a = 0, the
 *              boundary; rows a >= 1 are -inf)
 * draft_ids    int32 [B, P] out: [boundary, c_1, .., c_{P-1}]
 * margin       fp64 [B] out (optional): the smallest gap between the best
 *              and the runner-up score over every max this request took
 */
int oracle_dflash2_select(const float* cand_logits, const int32_t* boundary,
                          const uint16_t* hidden, const uint16_t* w_h,
                          const uint16_t* code_a, const uint16_t* code_b,
                          int32_t batch, int32_t positions, int64_t vocab,
                          int32_t top, int32_t rank, int32_t dim, int32_t mode,
                          int32_t* cand_ids, double* cand_logit, double* trans,
                          int32_t* draft_ids, double* margin,
                          int32_t nthreads) {
  if (batch < 0 || positions < 2 || positions > 16 || top < 1 || top > 16 ||
      rank < 1 || dim < 1 || vocab < top || (mode != 0 && mode != 1))
    return ORACLE_ERR_ARG;
  const int P1 = positions - 1, K = top;
  int err = ORACLE_OK;
#ifdef _OPENMP
  if (nthreads < 1) nthreads = omp_get_max_threads();
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
#endif
  for (int b = 0; b < batch; ++b) {
    double* hh = (double*)malloc(sizeof(double) * (size_t)rank);
    if (!hh) {
#ifdef _OPENMP
#pragma omp critical
#endif
      err = ORACLE_ERR_NOMEM;
      continue;
    }
    double mg = INFINITY;
    int32_t* ci = cand_ids + (int64_t)b * P1 * K;
    double* cl = cand_logit + (int64_t)b * P1 * K;
    double* tr = trans + (int64_t)b * P1 * K * K;
    for (int t = 1; t <= P1; ++t) {
      /* candidates of position t */
      int32_t ids[16];
      float vals[16];
      top_k(cand_logits + ((int64_t)b * P1 + t - 1) * vocab, vocab, K, ids, vals);
      for (int i = 0; i < K; ++i) {
        ci[(t - 1) * K + i] = ids[i];
        cl[(t - 1) * K + i] = (double)vals[i];
      }
      /* H_t = W_H h_t */
      const uint16_t* h = hidden + ((int64_t)b * P1 + t - 1) * dim;
      for (int r = 0; r < rank; ++r) {
        double acc = 0.0;
        for (int d = 0; d < dim; ++d)
          acc += oracle_bf16_to_double(w_h[(int64_t)r * dim + d]) *
                 oracle_bf16_to_double(h[d]);
        hh[r] = acc;
      }
      /* S_t(a, c) for every predecessor rank a and successor rank c */
      const int n_pred = t == 1 ? 1 : K;
      for (int a = 0; a < K; ++a) {
        for (int c = 0; c < K; ++c) {
          double s = -INFINITY;
          if (a < n_pred) {
            const int32_t ta = t == 1 ? boundary[b] : ci[(t - 2) * K + a];
            const int32_t tc = ci[(t - 1) * K + c];
            s = cl[(t - 1) * K + c];
            for (int r = 0; r < rank; ++r)
              s += oracle_bf16_to_double(code_a[(int64_t)ta * rank + r]) * hh[r] *
                   oracle_bf16_to_double(code_b[(int64_t)tc * rank + r]);
          }
          tr[((int64_t)(t - 1) * K + a) * K + c] = s;
        }
      }
    }
    /* the walk */
    int32_t* out = draft_ids + (int64_t)b * positions;
    out[0] = boundary[b];
    if (mode == ORACLE_SELECT_GREEDY) {
      int prev = 0; /* rank of the chosen predecessor (the boundary at t=1) */
      for (int t = 1; t <= P1; ++t) {
        const double* row = tr + ((int64_t)(t - 1) * K + prev) * K;
        int best = 0;
        double second = -INFINITY;
        for (int c = 1; c < K; ++c) {
          if (row[c] > row[best]) {
            if (row[best] > second) second = row[best];
            best = c;
          } else if (row[c] > second) {
            second = row[c];
          }
        }
        if (row[best] - second < mg) mg = row[best] - second;
        out[t] = ci[(t - 1) * K + best];
        prev = best;
      }
    } else {
      /* exact MAP: best[t][c] = max_a best[t-1][a] + S_t(a, c) */
      double best[16][16];
      int back[16][16];
      for (int c = 0; c < K; ++c) {
        best[1][c] = tr[(int64_t)0 * K * K + 0 * K + c];
        back[1][c] = 0;
      }
      for (int t = 2; t <= P1; ++t) {
        for (int c = 0; c < K; ++c) {
          int arg = 0;
          double v = best[t - 1][0] + tr[((int64_t)(t - 1) * K + 0) * K + c];
          double second = -INFINITY;
          for (int a = 1; a < K; ++a) {
            const double w = best[t - 1][a] + tr[((int64_t)(t - 1) * K + a) * K + c];
            if (w > v) {
              if (v > second) second = v;
              v = w;
              arg = a;
            } else if (w > second) {
              second = w;
            }
          }
          best[t][c] = v;
          back[t][c] = arg;
          if (v - second < mg) mg = v - second;
        }
      }
      int c = 0;
      double second = -INFINITY;
      for (int i = 1; i < K; ++i) {
        if (best[P1][i] > best[P1][c]) {
          if (best[P1][c] > second) second = best[P1][c];
          c = i;
        } else if (best[P1][i] > second) {
          second = best[P1][i];
        }
      }
      if (best[P1][c] - second < mg) mg = best[P1][c] - second;
      for (int t = P1; t >= 1; --t) {
        out[t] = ci[(t - 1) * K + c];
        c = back[t][c];
      }
    }
    if (margin) margin[b] = mg;
    free(hh);
  }
  return err;
}
