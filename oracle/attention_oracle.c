/*
 * attention_oracle.c — the CPU oracle for attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this.  It shares no code, header, table or helper
 * with the CUDA library, and the CUDA library never calls it.
 *
 * What it computes, and where that is defined
 * -------------------------------------------
 * "vLLM Cascade Attention：用法、场景与原理解析" (beaiera.top):
 *   §一  cascade splits attention into a prefix phase (all queries, non-causal,
 *        over the shared KV), a suffix phase (each request, causal, over its own
 *        KV) and an LSE merge, and is mathematically equal to standard attention.
 *   §四  the worked example R1/R2: the KV of a request holds the tokens already
 *        computed plus this step's query tokens; the query tokens are the last
 *        q_len positions of the request's KV.
 *   §五, §十  the standard path: every request attends over its full KV, read
 *        page by page through block_table[seq_id].
 *   §八 Step 5  prefix phase = non-causal over KV [0, common_prefix_len) through
 *        block_table row 0; suffix phase = causal over KV [common_prefix_len,
 *        seq_len); merge = LSE rescaling (merge_attn_states).
 *
 * The oracle is the plain definition: for request r, query token i (absolute
 * position p = seq_len_r - q_len_r + i, the bottom-right causal alignment the
 * §四 example implies), query head h (KV head g = h / (Hq/Hkv)):
 *     s_j   = scale * sum_d q[d] * k_j[d]                  for keys j in the range
 *     lse   = m + ln(sum_j exp(s_j - m)),  m = max_j s_j   (natural log)
 *     out   = sum_j exp(s_j - m) v_j / sum_j exp(s_j - m)
 * Key range: FULL = [0, p] (the standard path), PREFIX = [0, cpl) (the prefix
 * phase), SUFFIX = [cpl, p] (the suffix phase).  Key j of request r lives in
 * physical block block_table[r][j / block_size], slot j % block_size.
 *
 * Attention sinks (§九 "Attention Sinks": a mechanism that always lets attention
 * put weight on a token outside the request's keys; every backend takes an optional
 * `sinks` argument).  Read as one logit s_h per query head, in natural-log units and
 * not multiplied by the scale, that joins the softmax of every row of head h as one
 * more key whose value row is zero.  Standard path only (a phase partial has none):
 *     m   = max(max_j s_j, s_h),   l = sum_j exp(s_j - m) + exp(s_h - m)
 *     out = sum_j exp(s_j - m) v_j / l,   lse = m + ln(l)
 * s_h = -inf is the standard path exactly.
 *
 * FP8 KV cache (§六: FlashInfer's cascade wrapper refuses a KV cache stored in FP8;
 * the page names the format, not its encoding).  Read as the OCP FP8 E4M3 format
 * ("e4m3fn": 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no
 * infinities, S.1111.111 = NaN, largest finite 448) with one scale per tensor, as
 * KV caches store it: an element's value is decode(byte) * k_scale (or * v_scale),
 *     decode = (-1)^S * 2^(E-7) * (1 + M/8)   for E > 0,
 *              (-1)^S * 2^-6 * (M/8)          for E = 0,
 * and attention runs on those values exactly as on a bf16 cache.
 *
 * Every floating-point step is IEEE double; bf16 inputs are widened exactly.
 * Sums run in key / feature index order.  No blocking, no fusion, no reordering.
 * An empty key range gives out = 0 and lse = -inf.
 *
 * Layouts (all row-major, contiguous):
 *   q        bf16 bits [total_q, Hq, D]
 *   k, v     bf16 bits [num_blocks, block_size, Hkv, D] (or E4M3 bytes, same shape)
 *   block_table int32 [num_reqs, bt_stride]   (only the first cdiv(seq_len, bs)
 *            entries of a row are read)
 *   cu_seqlens_q int32 [num_reqs + 1], seq_lens int32 [num_reqs]
 *   out      double [n_rows, D] in (token, head) order, lse double [n_rows]
 *
 * Test-only fault planting: compiling with -DORACLE_MUTANT=<n> builds a copy
 * with one deliberate mistake, so the tests can show that their pins catch it.
 * The normal build (no macro) contains none of them.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

enum { ORACLE_FULL = 0, ORACLE_PREFIX = 1, ORACLE_SUFFIX = 2 };

typedef struct {
  const uint16_t* q;
  const void* k;
  const void* v;
  int32_t num_blocks;
  int32_t block_size;
  const int32_t* block_table;
  int64_t bt_stride;
  const int32_t* cu_seqlens_q;
  const int32_t* seq_lens;
  int32_t num_reqs;
  int32_t Hq, Hkv, D;
  double scale;
  int32_t mode;
  int32_t cpl;
  const double* sinks; /* [Hq] or NULL: no sinks (standard path only) */
  int32_t kv_fp8;      /* 0: k, v are bf16 bits; 1: E4M3 bytes with the scales below */
  double k_scale, v_scale;
} oracle_problem;

/* The E4M3 byte b as a double, from the format's definition (header). */
static double e4m3_to_double(uint8_t b) {
  const int sign = b >> 7;
  const int e = (b >> 3) & 15;
  const int mant = b & 7;
  if (e == 15 && mant == 7) return NAN;
#if ORACLE_MUTANT == 9
  const double mag = e == 0 ? ldexp(mant / 8.0, -6) : ldexp(1.0 + mant / 8.0, e - 8); /* planted: bias 8 */
#else
  const double mag = e == 0 ? ldexp(mant / 8.0, -6) : ldexp(1.0 + mant / 8.0, e - 7);
#endif
  return sign ? -mag : mag;
}

/* oracle_e4m3_decode: the 256 codes' values (for the tests' pins). */
void oracle_e4m3_decode(double* out256) {
  for (int b = 0; b < 256; ++b) out256[b] = e4m3_to_double((uint8_t)b);
}

static double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Request that owns global query token t: cu_seqlens_q[r] <= t < cu_seqlens_q[r+1]. */
static int request_of_token(const oracle_problem* P, int32_t t) {
  for (int r = 0; r < P->num_reqs; ++r)
    if (t >= P->cu_seqlens_q[r] && t < P->cu_seqlens_q[r + 1]) return r;
  return -1;
}

/* Element d of a K or V row: bf16 widened, or an E4M3 byte decoded and scaled. */
static double kv_elem(const oracle_problem* P, const void* row, int d, double scale) {
  if (P->kv_fp8) return e4m3_to_double(((const uint8_t*)row)[d]) * scale;
  return bf16_bits_to_double(((const uint16_t*)row)[d]);
}

/* Address of the D features of logical key j of request r, KV head g. */
static const void* kv_row(const oracle_problem* P, const void* cache, int r, int32_t j, int g,
                          int* bad) {
#if ORACLE_MUTANT == 5
  int32_t blk = P->block_table[(int64_t)r * P->bt_stride + j / P->block_size];
  int32_t slot = (j + 1) % P->block_size; /* planted: slot off by one inside the page */
#else
  int32_t blk = P->block_table[(int64_t)r * P->bt_stride + j / P->block_size];
  int32_t slot = j % P->block_size;
#endif
  if (blk < 0 || blk >= P->num_blocks || slot < 0 || slot >= P->block_size) {
    *bad = 1;
    return NULL;
  }
  const int64_t elem = (((int64_t)blk * P->block_size + slot) * P->Hkv + g) * (int64_t)P->D;
  return (const uint8_t*)cache + elem * (P->kv_fp8 ? 1 : 2);
}

/* One output row: query token t, query head h.  Returns 0, or -1 on a bad index. */
static int attend_row(const oracle_problem* P, int32_t t, int32_t h, double* out, double* lse) {
  const int r = request_of_token(P, t);
  if (r < 0 || h < 0 || h >= P->Hq) return -1;
  const int32_t q_len = P->cu_seqlens_q[r + 1] - P->cu_seqlens_q[r];
  const int32_t i = t - P->cu_seqlens_q[r];
  const int32_t pos = P->seq_lens[r] - q_len + i; /* absolute position of the query */
  const int group = P->Hq / P->Hkv;
#if ORACLE_MUTANT == 3
  const int g = h % P->Hkv; /* planted: interleaved instead of contiguous GQA groups */
#else
  const int g = h / group;
#endif
  int32_t lo, hi; /* key range [lo, hi) */
  if (P->mode == ORACLE_PREFIX) {
    lo = 0;
    hi = P->cpl;
  } else if (P->mode == ORACLE_SUFFIX) {
    lo = P->cpl;
    hi = pos + 1;
  } else {
    lo = 0;
#if ORACLE_MUTANT == 2
    hi = pos; /* planted: the query does not see its own key */
#else
    hi = pos + 1;
#endif
  }
  const int D = P->D;
  /* the sink logit of this row's head (standard path only); -inf: none */
  const double sink = (P->sinks && P->mode == ORACLE_FULL) ? P->sinks[h] : -INFINITY;
  if (hi <= lo) {
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    *lse = sink;
    return 0;
  }
  const uint16_t* qrow = P->q + ((int64_t)t * P->Hq + h) * D;
  double* s = (double*)malloc(sizeof(double) * (size_t)(hi - lo));
  if (!s) return -1;
  int bad = 0;
  double m = -INFINITY;
  for (int32_t j = lo; j < hi; ++j) {
    const void* krow = kv_row(P, P->k, r, j, g, &bad);
    if (bad) {
      free(s);
      return -1;
    }
    double acc = 0.0;
    for (int d = 0; d < D; ++d)
      acc += bf16_bits_to_double(qrow[d]) * kv_elem(P, krow, d, P->k_scale);
#if ORACLE_MUTANT == 1
    s[j - lo] = acc; /* planted: softmax scale dropped */
#else
    s[j - lo] = P->scale * acc;
#endif
    if (s[j - lo] > m) m = s[j - lo];
  }
  if (sink > m) m = sink;
  double l = 0.0;
  for (int32_t j = lo; j < hi; ++j) l += exp(s[j - lo] - m);
#if ORACLE_MUTANT == 8
  l += exp(m - sink); /* planted: the sink's exponent with its sign flipped */
#else
  if (sink != -INFINITY) l += exp(sink - m);
#endif
  for (int d = 0; d < D; ++d) {
    double acc = 0.0;
    for (int32_t j = lo; j < hi; ++j) {
      const void* vrow = kv_row(P, P->v, r, j, g, &bad);
      if (bad) {
        free(s);
        return -1;
      }
#if ORACLE_MUTANT == 6
      acc += exp(s[j - lo] - m) * kv_elem(P, vrow, (d + 1) % D, P->v_scale); /* planted: feature shift */
#else
      acc += exp(s[j - lo] - m) * kv_elem(P, vrow, d, P->v_scale);
#endif
    }
    out[d] = acc / l;
  }
#if ORACLE_MUTANT == 4
  *lse = (m + log(l)) / log(2.0); /* planted: base-2 instead of natural log */
#else
  *lse = m + log(l);
#endif
  free(s);
  return 0;
}

typedef struct {
  const oracle_problem* P;
  const int32_t* row_token;
  const int32_t* row_head;
  int64_t first, last; /* rows [first, last) */
  double* out;
  double* lse;
  int status;
} oracle_job;

static void* run_job(void* arg) {
  oracle_job* J = (oracle_job*)arg;
  J->status = 0;
  for (int64_t n = J->first; n < J->last; ++n) {
    int32_t t, h;
    if (J->row_token) {
      t = J->row_token[n];
      h = J->row_head[n];
    } else {
      t = (int32_t)(n / J->P->Hq);
      h = (int32_t)(n % J->P->Hq);
    }
    if (attend_row(J->P, t, h, J->out + n * J->P->D, J->lse + n) != 0) J->status = -1;
  }
  return NULL;
}

static int run_rows(const oracle_problem* P, const int32_t* row_token, const int32_t* row_head,
                    int64_t n_rows, double* out, double* lse, int n_threads) {
  if (P->Hkv <= 0 || P->Hq <= 0 || P->Hq % P->Hkv != 0 || P->D <= 0 || P->block_size <= 0)
    return -2;
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  if (n_rows < n_threads) n_threads = n_rows > 0 ? (int)n_rows : 1;
  oracle_job jobs[256];
  pthread_t tid[256];
  int64_t per = (n_rows + n_threads - 1) / n_threads;
  for (int i = 0; i < n_threads; ++i) {
    jobs[i].P = P;
    jobs[i].row_token = row_token;
    jobs[i].row_head = row_head;
    jobs[i].first = (int64_t)i * per < n_rows ? (int64_t)i * per : n_rows;
    jobs[i].last = (int64_t)(i + 1) * per < n_rows ? (int64_t)(i + 1) * per : n_rows;
    jobs[i].out = out;
    jobs[i].lse = lse;
    jobs[i].status = 0;
  }
  if (n_threads == 1) {
    run_job(&jobs[0]);
    return jobs[0].status;
  }
  for (int i = 0; i < n_threads; ++i) pthread_create(&tid[i], NULL, run_job, &jobs[i]);
  int status = 0;
  for (int i = 0; i < n_threads; ++i) {
    pthread_join(tid[i], NULL);
    if (jobs[i].status) status = jobs[i].status;
  }
  return status;
}

/*
 * oracle_attention: every (token, head) row of the batch, in [total_q, Hq] order.
 * mode: 0 = standard path (keys [0, p]), 1 = prefix phase (keys [0, cpl),
 * non-causal), 2 = suffix phase (keys [cpl, p]).  Returns 0, -1 on an
 * out-of-range block id, -2 on bad shapes.
 */
int oracle_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, int32_t num_blocks,
                     int32_t block_size, const int32_t* block_table, int64_t bt_stride,
                     const int32_t* cu_seqlens_q, const int32_t* seq_lens, int32_t num_reqs,
                     int32_t Hq, int32_t Hkv, int32_t D, double scale, int32_t mode, int32_t cpl,
                     double* out, double* lse, int32_t n_threads) {
  oracle_problem P = {q,           k,        v,    num_blocks, block_size, block_table, bt_stride,
                      cu_seqlens_q, seq_lens, num_reqs, Hq,  Hkv,        D,           scale,
                      mode,        cpl,      NULL, 0, 1.0, 1.0};
  int64_t total_q = cu_seqlens_q[num_reqs];
  return run_rows(&P, NULL, NULL, total_q * Hq, out, lse, n_threads);
}

/* oracle_attention_sinks: the standard path with per-head sinks (sinks [Hq]). */
int oracle_attention_sinks(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           int32_t num_blocks, int32_t block_size, const int32_t* block_table,
                           int64_t bt_stride, const int32_t* cu_seqlens_q, const int32_t* seq_lens,
                           int32_t num_reqs, int32_t Hq, int32_t Hkv, int32_t D, double scale,
                           const double* sinks, const int32_t* row_token, const int32_t* row_head,
                           int64_t n_rows, double* out, double* lse, int32_t n_threads) {
  oracle_problem P = {q,           k,        v,    num_blocks, block_size, block_table, bt_stride,
                      cu_seqlens_q, seq_lens, num_reqs, Hq,  Hkv,        D,           scale,
                      ORACLE_FULL, 0,       sinks, 0, 1.0, 1.0};
  if (row_token) return run_rows(&P, row_token, row_head, n_rows, out, lse, n_threads);
  return run_rows(&P, NULL, NULL, (int64_t)cu_seqlens_q[num_reqs] * Hq, out, lse, n_threads);
}

/* oracle_attention_rows: only the listed (token, head) rows, for sampled checks. */
int oracle_attention_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          int32_t num_blocks, int32_t block_size, const int32_t* block_table,
                          int64_t bt_stride, const int32_t* cu_seqlens_q, const int32_t* seq_lens,
                          int32_t num_reqs, int32_t Hq, int32_t Hkv, int32_t D, double scale,
                          int32_t mode, int32_t cpl, const int32_t* row_token,
                          const int32_t* row_head, int64_t n_rows, double* out, double* lse,
                          int32_t n_threads) {
  oracle_problem P = {q,           k,        v,    num_blocks, block_size, block_table, bt_stride,
                      cu_seqlens_q, seq_lens, num_reqs, Hq,  Hkv,        D,           scale,
                      mode,        cpl,      NULL, 0, 1.0, 1.0};
  return run_rows(&P, row_token, row_head, n_rows, out, lse, n_threads);
}

/*
 * oracle_attention_fp8kv: the listed rows (row_token NULL: every row, [total_q, Hq]
 * order) over an E4M3 KV cache with per-tensor scales, in any mode.
 */
int oracle_attention_fp8kv(const uint16_t* q, const uint8_t* k, const uint8_t* v,
                           int32_t num_blocks, int32_t block_size, const int32_t* block_table,
                           int64_t bt_stride, const int32_t* cu_seqlens_q, const int32_t* seq_lens,
                           int32_t num_reqs, int32_t Hq, int32_t Hkv, int32_t D, double scale,
                           double k_scale, double v_scale, int32_t mode, int32_t cpl,
                           const int32_t* row_token, const int32_t* row_head, int64_t n_rows,
                           double* out, double* lse, int32_t n_threads) {
  oracle_problem P = {q,           k,        v,    num_blocks, block_size, block_table, bt_stride,
                      cu_seqlens_q, seq_lens, num_reqs, Hq,  Hkv,        D,           scale,
                      mode,        cpl,      NULL, 1, k_scale, v_scale};
  if (row_token) return run_rows(&P, row_token, row_head, n_rows, out, lse, n_threads);
  return run_rows(&P, NULL, NULL, (int64_t)cu_seqlens_q[num_reqs] * Hq, out, lse, n_threads);
}

/*
 * oracle_merge_states: the LSE merge of two partial results (merge_attn_states,
 * "vLLM Cascade Attention：用法、场景与原理解析" §一 and §八 Step 5):
 *     m = max(l1, l2),  w1 = exp(l1 - m),  w2 = exp(l2 - m)
 *     out = (w1 o1 + w2 o2) / (w1 + w2),   lse = m + ln(w1 + w2)
 * Both partials empty (l1 = l2 = -inf): out = 0, lse = -inf.
 */
void oracle_merge_states(const double* o1, const double* l1, const double* o2, const double* l2,
                         int64_t n_rows, int32_t D, double* out, double* lse) {
  for (int64_t n = 0; n < n_rows; ++n) {
    const double a = l1[n], b = l2[n];
    if (a == -INFINITY && b == -INFINITY) {
      for (int d = 0; d < D; ++d) out[n * D + d] = 0.0;
      lse[n] = -INFINITY;
      continue;
    }
    const double m = a > b ? a : b;
    const double w1 = exp(a - m);
#if ORACLE_MUTANT == 7
    const double w2 = exp(m - b); /* planted: sign of the second exponent flipped */
#else
    const double w2 = exp(b - m);
#endif
    for (int d = 0; d < D; ++d) out[n * D + d] = (w1 * o1[n * D + d] + w2 * o2[n * D + d]) / (w1 + w2);
    lse[n] = m + log(w1 + w2);
  }
}

/* Build identification for the loader (mutant number, 0 for the real oracle). */
int oracle_mutant_id(void) { return ORACLE_MUTANT; }
