/*
 * Paged GQA decode attention: plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may call, link or
 * load this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it. It shares no code, header or table with the CUDA path.
 *
 * What it computes (the plain definition of single-token decode attention):
 *   for request b, query head h, KV head g = h / (Hq / Hkv):
 *     A_b   = attended token positions: [0, L_b)            (global layer)
 *                                        [max(0, L_b - W), L_b) (window W > 0)
 *     K_b[t] = k_pool[block_table[b][t / P], g, t % P, :]   (V alike; V = K when
 *                                                            the layer shares K=V)
 *     s_t   = scale * sum_d q[b,h,d] * K_b[t,d]
 *     p_t   = exp(s_t - max s) / sum_{A_b} exp(s - max s)
 *     o     = sum_{t in A_b} p_t * V_b[t,:]
 *   and o = 0 when A_b is empty.
 *
 * Sources (page title, section):
 *   - decode = attention of one new token over the cached keys/values:
 *     "模型库与算子层 — 概念" (vLLM model library & operator layer, concepts),
 *     section "注意力层 / 核心操作" (attention layer, core operations);
 *   - the paged KV cache, logical layout [L, B, H, N, C] and block sizes that are
 *     multiples of 16: same page, "KV-Cache 布局统一" (KV-cache layout) and the
 *     block-size paragraph of "核心操作";
 *   - several query heads share one KV head (GQA), sliding-window layers and
 *     global layers with their own head_dim / KV-head count, and K=V storage:
 *     Sparse-vLLM PR #27 "feat: support Gemma 4 and native multimodal
 *     inference", sections "Gemma 4 文本推理" (text inference) and
 *     "专用算子与性能优化" (dedicated operators);
 *   - the split-KV partial results with a log-sum-exp slot, merged afterwards:
 *     vLLM concepts page, section "MLA 与 Sparse MLA（DSA）" (MLA decode);
 *   - an FP8 KV cache (the same decode over e4m3 values times per-(page, KV
 *     head) scales): the vLLM concepts page records FP8 KV-cache support in its
 *     Blackwell (SM100) FlashAttention-4 backend (section "JIT 预热基础设施") and a
 *     Blackwell sparse-MLA backend that takes an FP8 KV cache (section "MLA 与
 *     Sparse MLA（DSA）"); the e4m3 format and the scale granularity are this
 *     library's reading.
 *
 * Readings where the pages are silent: the window keeps exactly the last W
 * positions including the current token; query head h uses KV head h / G; the
 * pool layout is [num_pages, Hkv, P, d] (the [B, H, N, C] slice of one layer).
 *
 * All arithmetic is IEEE fp64 from the exact bf16 (or e4m3 x fp32 scale) input
 * values. Build with
 * -ffp-contract=off so x86 and Arm hosts produce identical bits.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Status codes returned by every entry point. */
#define REF_OK 0
#define REF_BAD_ARG -1
#define REF_BAD_PAGE -2
#define REF_BAD_LEN -3
#define REF_NO_MEM -4

/* bf16 -> fp64: a bf16 value is the top 16 bits of an IEEE binary32. */
static double bf16_to_f64(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/*
 * OCP FP8 E4M3 ("fn" flavour: no infinities; S.1111.111 is the only NaN) ->
 * fp64, from the format's definition: 1 sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits; exponent field 0 encodes the subnormals m * 2^-9.
 */
static double e4m3_to_f64(uint8_t x) {
  const int sign = x >> 7, e = (x >> 3) & 15, m = x & 7;
  if (e == 15 && m == 7) return NAN;
  const double v = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -v : v;
}

typedef struct {
  int B, Hq, Hkv, d, P, num_pages, max_pages;
  const uint16_t *q, *k_pool, *v_pool; /* v_pool == NULL: V is K (K=V layer) */
  const int32_t *block_tables, *seq_lens;
  int window; /* 0 = global layer */
  double scale;
  /* FP8 KV cache: e4m3 pools with one scale per (page, KV head) for K and for V
   * (k8/v8 replace k_pool/v_pool; v8 == NULL: V is K, with K's scales) */
  int kv_fp8;
  const uint8_t *k8, *v8;
  const float *k_scale, *v_scale; /* [num_pages, Hkv] */
} ref_layer;

static int check_layer(const ref_layer *ly) {
  if (ly->B < 0 || ly->Hq <= 0 || ly->Hkv <= 0 || ly->d <= 0 || ly->P <= 0) return REF_BAD_ARG;
  if (ly->Hq % ly->Hkv != 0) return REF_BAD_ARG;
  if (ly->window < 0 || ly->num_pages < 0 || ly->max_pages < 0) return REF_BAD_ARG;
  if (ly->B > 0 && (!ly->q || !ly->block_tables || !ly->seq_lens)) return REF_BAD_ARG;
  if (ly->B > 0 && !ly->kv_fp8 && !ly->k_pool) return REF_BAD_ARG;
  if (ly->B > 0 && ly->kv_fp8 && (!ly->k8 || !ly->k_scale || (ly->v8 && !ly->v_scale))) return REF_BAD_ARG;
  for (int b = 0; b < ly->B; ++b) {
    int L = ly->seq_lens[b];
    if (L < 0 || (long long)L > (long long)ly->max_pages * ly->P) return REF_BAD_LEN;
  }
  return REF_OK;
}

/* Attended range [lo, hi) of request b. */
static void attended_range(const ref_layer *ly, int b, int *lo, int *hi) {
  int L = ly->seq_lens[b];
  *hi = L;
  *lo = (ly->window > 0 && L > ly->window) ? L - ly->window : 0;
}

/* The d values of token t of request b, KV head g, from the K (which = 0) or
 * V (which = 1) pool, widened to fp64 into row[0..d) (FP8 pools: the e4m3
 * value times its (page, KV head) scale). REF_BAD_PAGE if the block table
 * names a page outside the pool. */
static int load_row(const ref_layer *ly, int which, int b, int g, int t, double *row) {
  int32_t page = ly->block_tables[(size_t)b * ly->max_pages + t / ly->P];
  if (page < 0 || page >= ly->num_pages) return REF_BAD_PAGE;
  const size_t r = ((size_t)page * ly->Hkv + g) * ly->P + (size_t)(t % ly->P);
  const size_t base = r * ly->d;
  if (!ly->kv_fp8) {
    const uint16_t *pool = (which == 1 && ly->v_pool) ? ly->v_pool : ly->k_pool;
    for (int i = 0; i < ly->d; ++i) row[i] = bf16_to_f64(pool[base + i]);
  } else {
    const int use_v = (which == 1 && ly->v8);
    const uint8_t *pool8 = use_v ? ly->v8 : ly->k8;
    const double s = (use_v ? ly->v_scale : ly->k_scale)[(size_t)page * ly->Hkv + g];
    for (int i = 0; i < ly->d; ++i) row[i] = e4m3_to_f64(pool8[base + i]) * s;
  }
  return REF_OK;
}

/*
 * Attention of query row qrow (query head h of request b) over the token
 * positions [lo, hi):
 * writes o[0..d) (normalised by the softmax denominator) and returns the
 * natural-log log-sum-exp of the scaled scores through *lse (-inf, o = 0 when
 * the range is empty).
 */
static int attend_range(const ref_layer *ly, int b, int h, const uint16_t *qrow, int lo, int hi, double *o,
                        double *lse, double *s /* scratch, >= hi - lo */, double *row /* scratch, d */) {
  const int G = ly->Hq / ly->Hkv;
  const int g = h / G;
  const int d = ly->d;

  for (int i = 0; i < d; ++i) o[i] = 0.0;
  if (hi <= lo) {
    *lse = -INFINITY;
    return REF_OK;
  }
  /* scores s_t = scale * <q, K_t> */
  double m = -INFINITY;
  for (int t = lo; t < hi; ++t) {
    if (load_row(ly, 0, b, g, t, row) != REF_OK) return REF_BAD_PAGE;
    double acc = 0.0;
    for (int i = 0; i < d; ++i) acc += bf16_to_f64(qrow[i]) * row[i];
    s[t - lo] = ly->scale * acc;
    if (s[t - lo] > m) m = s[t - lo];
  }
  /* softmax weights exp(s - max) and their sum */
  double l = 0.0;
  for (int t = lo; t < hi; ++t) {
    s[t - lo] = exp(s[t - lo] - m);
    l += s[t - lo];
  }
  /* weighted sum of the value rows */
  for (int t = lo; t < hi; ++t) {
    if (load_row(ly, 1, b, g, t, row) != REF_OK) return REF_BAD_PAGE;
    const double p = s[t - lo];
    for (int i = 0; i < d; ++i) o[i] += p * row[i];
  }
  for (int i = 0; i < d; ++i) o[i] /= l;
  *lse = m + log(l);
  return REF_OK;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
}

static int max_seq_len(const ref_layer *ly) {
  int max_len = 0;
  for (int b = 0; b < ly->B; ++b) max_len = ly->seq_lens[b] > max_len ? ly->seq_lens[b] : max_len;
  return max_len;
}

/* Rows (b * Hq + h) of the decode, in parallel over rows. */
static int decode_rows(const ref_layer *ly, const int32_t *rows, int n_rows, double *out, double *lse_out,
                       int nthreads) {
  int st = check_layer(ly);
  if (st != REF_OK) return st;
  if (!out) return REF_BAD_ARG;
  const int B = ly->B, Hq = ly->Hq, d = ly->d;
  const int total = rows ? n_rows : B * Hq;
  const int max_len = max_seq_len(ly);

  int status = REF_OK;
  set_threads(nthreads);
#pragma omp parallel
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    double *row = (double *)malloc(sizeof(double) * (size_t)d);
    if (!s || !row) {
#pragma omp critical
      status = REF_NO_MEM;
    }
#pragma omp for schedule(dynamic, 1)
    for (int r = 0; r < total; ++r) {
      if (!s || !row) continue;
      const int rix = rows ? rows[r] : r;
      if (rix < 0 || rix >= B * Hq) {
#pragma omp critical
        status = REF_BAD_ARG;
        continue;
      }
      const int b = rix / Hq, h = rix % Hq;
      int lo, hi;
      attended_range(ly, b, &lo, &hi);
      double lse;
      int rs = attend_range(ly, b, h, ly->q + (size_t)rix * d, lo, hi, out + (size_t)rix * d, &lse, s, row);
      if (lse_out) lse_out[rix] = lse;
      if (rs != REF_OK) {
#pragma omp critical
        status = rs;
      }
    }
    free(s);
    free(row);
  }
  return status;
}

/*
 * Full decode: out[b, h, :] for every request and query head (fp64), and the
 * log-sum-exp of each row into lse_out[b, h] when lse_out is not NULL.
 * Rows are listed by (b, h); `rows`/`n_rows` restrict the work to a subset
 * (each entry b * Hq + h); pass rows = NULL for all B * Hq rows. Output rows
 * not in the subset are left untouched.
 */
int ref_decode_rows(int B, int Hq, int Hkv, int d, int P, int num_pages, int max_pages,
                    const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                    const int32_t *block_tables, const int32_t *seq_lens, int window, double scale,
                    const int32_t *rows, int n_rows, double *out, double *lse_out, int nthreads) {
  ref_layer ly = {B, Hq, Hkv, d, P, num_pages, max_pages, q, k_pool, v_pool,
                  block_tables, seq_lens, window, scale, 0, NULL, NULL, NULL, NULL};
  return decode_rows(&ly, rows, n_rows, out, lse_out, nthreads);
}

/*
 * The same decode over an FP8 KV cache: k8 / v8 hold e4m3 bytes in the pool
 * layout [num_pages, Hkv, P, d], k_scale / v_scale one fp32 scale per
 * (page, KV head); the cached value is the e4m3 value times its scale. v8 =
 * NULL: V is K (K=V layer), with K's scales. q stays bf16.
 */
int ref_decode_rows_fp8(int B, int Hq, int Hkv, int d, int P, int num_pages, int max_pages,
                        const uint16_t *q, const uint8_t *k8, const uint8_t *v8, const float *k_scale,
                        const float *v_scale, const int32_t *block_tables, const int32_t *seq_lens, int window,
                        double scale, const int32_t *rows, int n_rows, double *out, double *lse_out,
                        int nthreads) {
  ref_layer ly = {B, Hq, Hkv, d, P, num_pages, max_pages, q, NULL, NULL,
                  block_tables, seq_lens, window, scale, 1, k8, v8, k_scale, v8 ? v_scale : NULL};
  return decode_rows(&ly, rows, n_rows, out, lse_out, nthreads);
}

/*
 * Several new tokens per request (speculative-decode verification, or a chunk
 * of prefill, over the paged cache): request b has T query tokens, the last T
 * of its L_b cached positions, all already in the cache. Query token j sits at
 * position pos_j = L_b - T + j and attends causally: positions [lo_j, pos_j]
 * with lo_j = 0 on a global layer and max(0, pos_j + 1 - W) on a window layer
 * (the last W positions up to and including its own) -- for every j, the
 * single-token decode of q[b, j] at length pos_j + 1.
 *   q [B, T, Hq, d] (bf16 bits), out [B, T, Hq, d] fp64, lse_out [B, T, Hq]
 *   (may be NULL). Returns REF_BAD_LEN if some L_b < T.
 * Sources: the pages reuse a paged prefill plan next to decode (Sparse-vLLM
 * PR #27, section "专用算子与性能优化") and list causal multi-token
 * verification for speculative decoding over a paged cache (vLLM concepts
 * page, section "MLA 与 Sparse MLA（DSA）").
 */
int ref_decode_multi(int B, int T, int Hq, int Hkv, int d, int P, int num_pages, int max_pages, const uint16_t *q,
                     const uint16_t *k_pool, const uint16_t *v_pool, const int32_t *block_tables,
                     const int32_t *seq_lens, int window, double scale, double *out, double *lse_out, int nthreads) {
  ref_layer ly = {B, Hq, Hkv, d, P, num_pages, max_pages, q, k_pool, v_pool,
                  block_tables, seq_lens, window, scale, 0, NULL, NULL, NULL, NULL};
  int st = check_layer(&ly);
  if (st != REF_OK) return st;
  if (T < 1 || !out) return REF_BAD_ARG;
  for (int b = 0; b < B; ++b)
    if (seq_lens[b] < T) return REF_BAD_LEN;
  const int max_len = max_seq_len(&ly);
  const int total = B * T * Hq;

  int status = REF_OK;
  set_threads(nthreads);
#pragma omp parallel
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    double *row = (double *)malloc(sizeof(double) * (size_t)d);
    if (!s || !row) {
#pragma omp critical
      status = REF_NO_MEM;
    }
#pragma omp for schedule(dynamic, 1)
    for (int r = 0; r < total; ++r) {
      if (!s || !row) continue;
      const int b = r / (T * Hq), j = (r / Hq) % T, h = r % Hq;
      const int pos = seq_lens[b] - T + j;
      const int hi = pos + 1;
      const int lo = (window > 0 && hi > window) ? hi - window : 0;
      double lse;
      int rs = attend_range(&ly, b, h, q + (size_t)r * d, lo, hi, out + (size_t)r * d, &lse, s, row);
      if (lse_out) lse_out[r] = lse;
      if (rs != REF_OK) {
#pragma omp critical
        status = rs;
      }
    }
    free(s);
    free(row);
  }
  return status;
}

/* e4m3 byte -> fp64 (exposed for the tests that pin the decoder). */
double ref_e4m3_to_f64(int x) { return e4m3_to_f64((uint8_t)x); }

/*
 * Split-KV first stage (vLLM concepts page, "MLA 与 Sparse MLA（DSA）"): the
 * attended range [lo, hi) of each request is cut into pieces of `chunk`
 * consecutive positions starting at lo; piece k covers
 * [lo + k * chunk, lo + (k + 1) * chunk) intersected with [lo, hi). Each piece
 * yields its normalised partial output o_part[b, h, k, :] and the log-sum-exp
 * lse_part[b, h, k] (-inf and zeros for an empty piece). num_splits pieces are
 * produced per row; pieces past the range are empty.
 */
int ref_decode_split(int B, int Hq, int Hkv, int d, int P, int num_pages, int max_pages,
                     const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                     const int32_t *block_tables, const int32_t *seq_lens, int window, double scale,
                     int num_splits, int chunk, double *o_part, double *lse_part, int nthreads) {
  ref_layer ly = {B, Hq, Hkv, d, P, num_pages, max_pages, q, k_pool, v_pool,
                  block_tables, seq_lens, window, scale, 0, NULL, NULL, NULL, NULL};
  int st = check_layer(&ly);
  if (st != REF_OK) return st;
  if (num_splits <= 0 || chunk <= 0 || !o_part || !lse_part) return REF_BAD_ARG;
  const int max_len = max_seq_len(&ly);

  int status = REF_OK;
  set_threads(nthreads);
#pragma omp parallel
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    double *rowbuf = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
    for (int row = 0; row < B * Hq; ++row) {
      if (!s || !rowbuf) continue;
      const int b = row / Hq, h = row % Hq;
      int lo, hi;
      attended_range(&ly, b, &lo, &hi);
      for (int k = 0; k < num_splits; ++k) {
        long long plo = (long long)lo + (long long)k * chunk;
        long long phi = plo + chunk;
        if (plo > hi) plo = hi;
        if (phi > hi) phi = hi;
        const size_t idx = (size_t)row * num_splits + k;
        int rs = attend_range(&ly, b, h, ly.q + ((size_t)b * Hq + h) * d, (int)plo, (int)phi, o_part + idx * d,
                              lse_part + idx, s, rowbuf);
        if (rs != REF_OK) {
#pragma omp critical
          status = rs;
        }
      }
    }
    if (!s || !rowbuf) {
#pragma omp critical
      status = REF_NO_MEM;
    }
    free(s);
    free(rowbuf);
  }
  return status;
}

/*
 * Split-KV second stage: merges the partial outputs of the pieces of each row
 * by their log-sum-exp weights,
 *   M = max_k lse_k,  w_k = exp(lse_k - M),  out = sum_k w_k o_k / sum_k w_k,
 * with out = 0 when every piece is empty (M = -inf).
 */
int ref_merge(int rows, int num_splits, int d, const double *o_part, const double *lse_part,
              double *out) {
  if (rows < 0 || num_splits <= 0 || d <= 0 || !o_part || !lse_part || !out) return REF_BAD_ARG;
  for (int r = 0; r < rows; ++r) {
    const double *lse = lse_part + (size_t)r * num_splits;
    double M = -INFINITY;
    for (int k = 0; k < num_splits; ++k)
      if (lse[k] > M) M = lse[k];
    double *o = out + (size_t)r * d;
    for (int i = 0; i < d; ++i) o[i] = 0.0;
    if (M == -INFINITY) continue;
    double wsum = 0.0;
    for (int k = 0; k < num_splits; ++k) {
      const double w = exp(lse[k] - M);
      wsum += w;
      const double *ok = o_part + ((size_t)r * num_splits + k) * d;
      for (int i = 0; i < d; ++i) o[i] += w * ok[i];
    }
    for (int i = 0; i < d; ++i) o[i] /= wsum;
  }
  return REF_OK;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int ref_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
