/*
 * paged_gqa_oracle.c -- plain fp64 CPU oracle for paged grouped-query attention.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load or run this file. It shares no code, header, table or
 * helper with the CUDA library; neither includes the other.
 *
 * What it computes (the plain definition, no blocking, fusion or reordering):
 *
 *   For every sequence s with q0 = query_start_loc[s], qn = query_start_loc[s+1]-q0,
 *   L = seq_lens[s], every query token t < qn and every query head h:
 *     kvh = h / (Hq/Hkv)                       contiguous head groups
 *     pos = L - qn + t                         bottom-right causal alignment
 *     qv[d]  = dec(q[q0+t, h, d]) * q_descale
 *     for every key j = 0..pos:
 *       b = block_table[s, j / P], r = j % P   the naive block-table walk
 *       kv[d] = dec(k_cache[b, r, kvh, d]) * k_descale
 *       vv[d] = dec(v_cache[b, r, kvh, d]) * v_descale
 *       s_j   = softmax_scale * sum_d qv[d] * kv[d]
 *     m = max_j s_j, w_j = exp(s_j - m)
 *     out[q0+t, h, d] = sum_j w_j vv_j[d] / sum_j w_j,  lse = m + log(sum_j w_j)
 *
 * Sources:
 *   - "Optimize Qwen3.5 MTP unified attention on gfx950" (sglang #36330): paged
 *     GQA attention over a block-tabled cache with separate K and V views, the
 *     kv-head index selecting the q-head group, per-tensor FP8 descale scalars
 *     (review thread and Modifications section).
 *   - "asm FP8 FMHA for prefix-hit prefill" (ROCm/ATOM #2534), summary: new
 *     tokens attend to cached plus new K/V, cu_seqlens_k longer than
 *     cu_seqlens_q, bottom-right causal mask.
 *   - OCP FP8 e4m3fn format: sign, 4 exponent bits with bias 7, 3 mantissa bits;
 *     normals (1+m/8)*2^(e-7), subnormals m*2^-9, S.1111.111 is NaN, no infinities.
 *   - bfloat16: the top 16 bits of an IEEE binary32.
 *
 * oracle_paged_gqa_sparse_attn (below) is the same row computation over a listed subset
 * of the keys ("Tune sparse GQA prefill profile on gfx942 and gfx950").
 *
 * Everything is fp64. exp/log are the C library's.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_BF16 = 1, OR_E4M3 = 3 };

enum {
  OR_OK = 0,
  OR_BAD_ARG = 1,        /* shapes, dtype, or qn > L                       */
  OR_BAD_BLOCK = 2,      /* a block-table entry the walk needs is out of range */
  OR_NO_MEMORY = 3
};

/* FP8 e4m3fn -> double, from the format definition. */
static double dec_e4m3(uint8_t x) {
  int sign = (x >> 7) & 1;
  int e = (x >> 3) & 0xF;
  int m = x & 0x7;
  double v;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);              /* m/8 * 2^(1-7) */
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

/* bfloat16 bits -> double: the bits are the high half of a binary32. */
static double dec_bf16(uint16_t x) {
  uint32_t u = (uint32_t)x << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* dec_e4m3 over all 256 codes, filled once before any parallel work. */
static double e4m3_value[256];

static void fill_e4m3_values(void) {
  for (int i = 0; i < 256; ++i) e4m3_value[i] = dec_e4m3((uint8_t)i);
}

static double dec(const void* base, int dtype, int64_t idx) {
  if (dtype == OR_E4M3) return e4m3_value[((const uint8_t*)base)[idx]];
  return dec_bf16(((const uint16_t*)base)[idx]);
}

/* Exposed so a test can compare the decode against an independent library. */
void oracle_e4m3_table(double* out256) {
  for (int i = 0; i < 256; ++i) out256[i] = dec_e4m3((uint8_t)i);
}

typedef struct {
  const void* q; int q_dtype; int64_t q_st, q_sh;                       /* [T, Hq, D]      */
  const void* k; const void* v; int kv_dtype;
  int64_t kv_sb, kv_sp, kv_sh;                                          /* [NB, P, Hkv, D] */
  const int32_t* block_table; int64_t bt_stride;
  const int32_t* seq_lens; const int32_t* qsl;
  int num_seqs, Hq, Hkv, D, P, NB;
  double q_descale, k_descale, v_descale, softmax_scale;
} oracle_args;

/* One output row (flat row = token*Hq + head). Returns an OR_ status. */
static int one_row(const oracle_args* a, int s, int t, int h, double* scores,
                   double* qv, double* o, double* lse_out) {
  const int G = a->Hq / a->Hkv;
  const int q0 = a->qsl[s];
  const int qn = a->qsl[s + 1] - q0;
  const int L = a->seq_lens[s];
  const int kvh = h / G;
  const int pos = L - qn + t;
  const int D = a->D;
  if (qn > L || pos < 0) return OR_BAD_ARG;

  /* the query row, dequantised */
  const int64_t qbase = (int64_t)(q0 + t) * a->q_st + (int64_t)h * a->q_sh;
  for (int d = 0; d < D; ++d) qv[d] = dec(a->q, a->q_dtype, qbase + d) * a->q_descale;

  /* scores */
  double m = -INFINITY;
  for (int j = 0; j <= pos; ++j) {
    int b = a->block_table[(int64_t)s * a->bt_stride + j / a->P];
    int r = j % a->P;
    if (b < 0 || b >= a->NB) return OR_BAD_BLOCK;
    int64_t kbase = (int64_t)b * a->kv_sb + (int64_t)r * a->kv_sp + (int64_t)kvh * a->kv_sh;
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += qv[d] * (dec(a->k, a->kv_dtype, kbase + d) * a->k_descale);
    scores[j] = a->softmax_scale * dot;
    if (scores[j] > m) m = scores[j];
  }

  /* softmax weights and the weighted sum of V */
  double l = 0.0;
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  for (int j = 0; j <= pos; ++j) {
    double w = exp(scores[j] - m);
    int b = a->block_table[(int64_t)s * a->bt_stride + j / a->P];
    int r = j % a->P;
    int64_t vbase = (int64_t)b * a->kv_sb + (int64_t)r * a->kv_sp + (int64_t)kvh * a->kv_sh;
    l += w;
    for (int d = 0; d < D; ++d) o[d] += w * dec(a->v, a->kv_dtype, vbase + d) * a->v_descale;
  }
  for (int d = 0; d < D; ++d) o[d] /= l;
  if (lse_out) *lse_out = m + log(l);
  return OR_OK;
}

/* Sequence index of a query token (query_start_loc is non-decreasing). */
static int seq_of_token(const oracle_args* a, int tok) {
  int lo = 0, hi = a->num_seqs - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if (a->qsl[mid] <= tok) lo = mid; else hi = mid - 1;
  }
  /* skip empty sequences that start at the same token */
  while (lo + 1 < a->num_seqs && a->qsl[lo + 1] <= tok) ++lo;
  return lo;
}

/*
 * Full or sampled evaluation.
 *   rows == NULL: every (token, head); out is [T, Hq, D], lse is [T, Hq] (optional).
 *   rows != NULL: the listed flat rows (token*Hq + head); out is [nrows, D],
 *                 lse is [nrows] (optional).
 * Returns 0, or the first non-zero OR_ status met.
 */
int oracle_paged_gqa_attn(const void* q, int q_dtype, int64_t q_st, int64_t q_sh,
                          const void* k, const void* v, int kv_dtype,
                          int64_t kv_sb, int64_t kv_sp, int64_t kv_sh,
                          const int32_t* block_table, int64_t bt_stride,
                          const int32_t* seq_lens, const int32_t* query_start_loc,
                          int num_seqs, int Hq, int Hkv, int D, int P, int NB,
                          double q_descale, double k_descale, double v_descale,
                          double softmax_scale, const int64_t* rows, int64_t nrows,
                          double* out, double* lse, int nthreads) {
  oracle_args a = {q, q_dtype, q_st, q_sh, k, v, kv_dtype, kv_sb, kv_sp, kv_sh,
                   block_table, bt_stride, seq_lens, query_start_loc,
                   num_seqs, Hq, Hkv, D, P, NB, q_descale, k_descale, v_descale, softmax_scale};
  if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || P <= 0) return OR_BAD_ARG;
  if ((q_dtype != OR_BF16 && q_dtype != OR_E4M3) || (kv_dtype != OR_BF16 && kv_dtype != OR_E4M3))
    return OR_BAD_ARG;
  if (num_seqs == 0) return OR_OK;
  const int64_t T = query_start_loc[num_seqs];
  int max_len = 1;
  for (int s = 0; s < num_seqs; ++s) {
    if (query_start_loc[s + 1] < query_start_loc[s]) return OR_BAD_ARG;
    if (query_start_loc[s + 1] - query_start_loc[s] > seq_lens[s]) return OR_BAD_ARG;
    if (seq_lens[s] > max_len) max_len = seq_lens[s];
  }
  const int64_t n = rows ? nrows : T * Hq;
  fill_e4m3_values();
  int status = OR_OK;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)max_len);
    double* o = (double*)malloc(sizeof(double) * (size_t)D);
    double* qv = (double*)malloc(sizeof(double) * (size_t)D);
    if (!scores || !o || !qv) {
#pragma omp critical
      status = OR_NO_MEMORY;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (int64_t i = 0; i < n; ++i) {
        int64_t flat = rows ? rows[i] : i;
        if (flat < 0 || flat >= T * Hq) {
#pragma omp critical
          status = status ? status : OR_BAD_ARG;
          continue;
        }
        int tok = (int)(flat / Hq), h = (int)(flat % Hq);
        int s = seq_of_token(&a, tok);
        double l_se = 0.0;
        int st = one_row(&a, s, tok - query_start_loc[s], h, scores, qv, o, &l_se);
        if (st != OR_OK) {
#pragma omp critical
          status = status ? status : st;
          continue;
        }
        memcpy(out + i * D, o, sizeof(double) * (size_t)D);
        if (lse) lse[i] = l_se;
      }
    }
    free(scores);
    free(o);
    free(qv);
  }
  return status;
}

/*
 * Sparse variant ("Tune sparse GQA prefill profile on gfx942 and gfx950", Overview and
 * Tests: each query row attends a selected list of tokens of its sequence, ~2k per row).
 * The list is given per (token, kv head) and shared by the kv head's G query heads:
 *
 *   for every listed entry p = indices[t, kvh, j], j = 0..K-1, with 0 <= p <= pos
 *   (pos = L - qn + t, the row's causal limit; other entries are not used):
 *     b = block_table[s, p / P], r = p % P
 *     s_j = softmax_scale * sum_d qv[d] * kv_p[d]
 *   out = sum_j exp(s_j - m) vv_p / sum_j exp(s_j - m) over the used entries (an entry
 *   listed twice counts twice); a row with no used entry is all zeros, lse = -inf.
 */
static int one_row_sparse(const oracle_args* a, int s, int t, int h, const int32_t* list, int K,
                          double* scores, double* qv, double* o, double* lse_out) {
  const int G = a->Hq / a->Hkv;
  const int q0 = a->qsl[s];
  const int qn = a->qsl[s + 1] - q0;
  const int L = a->seq_lens[s];
  const int kvh = h / G;
  const int pos = L - qn + t;
  const int D = a->D;
  if (qn > L || pos < 0) return OR_BAD_ARG;
  const int64_t qbase = (int64_t)(q0 + t) * a->q_st + (int64_t)h * a->q_sh;
  for (int d = 0; d < D; ++d) qv[d] = dec(a->q, a->q_dtype, qbase + d) * a->q_descale;
  double m = -INFINITY;
  int used = 0;
  for (int j = 0; j < K; ++j) {
    const int p = list[j];
    if (p < 0 || p > pos) continue;
    int b = a->block_table[(int64_t)s * a->bt_stride + p / a->P];
    if (b < 0 || b >= a->NB) return OR_BAD_BLOCK;
    int64_t kbase = (int64_t)b * a->kv_sb + (int64_t)(p % a->P) * a->kv_sp + (int64_t)kvh * a->kv_sh;
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += qv[d] * (dec(a->k, a->kv_dtype, kbase + d) * a->k_descale);
    scores[j] = a->softmax_scale * dot;
    if (scores[j] > m) m = scores[j];
    ++used;
  }
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  if (used == 0) {
    if (lse_out) *lse_out = -INFINITY;
    return OR_OK;
  }
  double l = 0.0;
  for (int j = 0; j < K; ++j) {
    const int p = list[j];
    if (p < 0 || p > pos) continue;
    const double w = exp(scores[j] - m);
    int b = a->block_table[(int64_t)s * a->bt_stride + p / a->P];
    int64_t vbase = (int64_t)b * a->kv_sb + (int64_t)(p % a->P) * a->kv_sp + (int64_t)kvh * a->kv_sh;
    l += w;
    for (int d = 0; d < D; ++d) o[d] += w * dec(a->v, a->kv_dtype, vbase + d) * a->v_descale;
  }
  for (int d = 0; d < D; ++d) o[d] /= l;
  if (lse_out) *lse_out = m + log(l);
  return OR_OK;
}

/* indices: [T, Hkv, K] int32 with strides (idx_st, idx_sh, 1). Rows and outputs as in
 * oracle_paged_gqa_attn. */
int oracle_paged_gqa_sparse_attn(const void* q, int q_dtype, int64_t q_st, int64_t q_sh,
                                 const void* k, const void* v, int kv_dtype,
                                 int64_t kv_sb, int64_t kv_sp, int64_t kv_sh,
                                 const int32_t* block_table, int64_t bt_stride,
                                 const int32_t* seq_lens, const int32_t* query_start_loc,
                                 const int32_t* indices, int64_t idx_st, int64_t idx_sh, int K,
                                 int num_seqs, int Hq, int Hkv, int D, int P, int NB,
                                 double q_descale, double k_descale, double v_descale,
                                 double softmax_scale, const int64_t* rows, int64_t nrows,
                                 double* out, double* lse, int nthreads) {
  oracle_args a = {q, q_dtype, q_st, q_sh, k, v, kv_dtype, kv_sb, kv_sp, kv_sh,
                   block_table, bt_stride, seq_lens, query_start_loc,
                   num_seqs, Hq, Hkv, D, P, NB, q_descale, k_descale, v_descale, softmax_scale};
  if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || P <= 0 || K < 0) return OR_BAD_ARG;
  if ((q_dtype != OR_BF16 && q_dtype != OR_E4M3) || (kv_dtype != OR_BF16 && kv_dtype != OR_E4M3))
    return OR_BAD_ARG;
  if (num_seqs == 0) return OR_OK;
  const int64_t T = query_start_loc[num_seqs];
  for (int s = 0; s < num_seqs; ++s) {
    if (query_start_loc[s + 1] < query_start_loc[s]) return OR_BAD_ARG;
    if (query_start_loc[s + 1] - query_start_loc[s] > seq_lens[s]) return OR_BAD_ARG;
  }
  const int64_t n = rows ? nrows : T * Hq;
  const int G = Hq / Hkv;
  fill_e4m3_values();
  int status = OR_OK;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    double* o = (double*)malloc(sizeof(double) * (size_t)D);
    double* qv = (double*)malloc(sizeof(double) * (size_t)D);
    if (!scores || !o || !qv) {
#pragma omp critical
      status = OR_NO_MEMORY;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (int64_t i = 0; i < n; ++i) {
        int64_t flat = rows ? rows[i] : i;
        if (flat < 0 || flat >= T * Hq) {
#pragma omp critical
          status = status ? status : OR_BAD_ARG;
          continue;
        }
        int tok = (int)(flat / Hq), h = (int)(flat % Hq);
        int s = seq_of_token(&a, tok);
        const int32_t* list = indices + (int64_t)tok * idx_st + (int64_t)(h / G) * idx_sh;
        double l_se = 0.0;
        int st = one_row_sparse(&a, s, tok - query_start_loc[s], h, list, K, scores, qv, o, &l_se);
        if (st != OR_OK) {
#pragma omp critical
          status = status ? status : st;
          continue;
        }
        memcpy(out + i * D, o, sizeof(double) * (size_t)D);
        if (lse) lse[i] = l_se;
      }
    }
    free(scores);
    free(o);
    free(qv);
  }
  return status;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
