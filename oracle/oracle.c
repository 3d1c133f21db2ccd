/*
 * oracle.c -- plain, slow, single-threaded CPU oracle for the batched
 * decode-step attention path (KV-cache scatter + softmax attention).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) may include, link or call this file.  Only the
 * tests, the smoke check and the benchmark's CPU-baseline leg use it.  It
 * shares no code, header, table or constant with the CUDA path.
 *
 * What it follows (the pages' text, restated):
 *   - realizar 0.8.5, src/cuda/executor/head_dim.rs, doc comment of
 *     `flash_decoding_attention_into` (PAR-118): Q is [M, num_heads,
 *     head_dim], the new K and V rows are [M, num_kv_heads, head_dim], the
 *     output is [M, num_heads, head_dim]; the KV cache is split into chunks
 *     processed independently and the partial results are merged with
 *     softmax rescaling.
 *   - same function, "Step 1: Scatter K/V to caches": every sequence's new
 *     K and V row is written into that sequence's cache at its position
 *     before attention runs; the per-sequence cache starts at
 *     seq_idx * batched_kv_stride and holds [num_kv_heads][max_len][head_dim].
 *   - same function, "Update cache lengths": a sequence at position p
 *     attends over p + 1 cache rows (rows 0..p inclusive).
 *   - same function, "Step 3: Compute max chunks needed": the number of
 *     chunks of a sequence is ceil(seq_len / chunk_size).
 *
 * The method (split-K with a rescaling merge) is exact up to rounding, so
 * the reference computation here is the plain definition of softmax
 * attention, evaluated in IEEE double:
 *     s_j = (1/sqrt(D)) * sum_d q[d] * K[j][d]            j = 0..L-1
 *     m   = max_j s_j,  w_j = exp(s_j - m),  Z = sum_j w_j
 *     o[d] = (sum_j w_j * V[j][d]) / Z
 * The split-K variant (oracle_attend_row_split) exists only so that tests
 * can pin the chunk-partial / rescaled-merge algebra against the definition.
 *
 * Readings of points the pages leave open (each also listed in the design
 * notes): softmax scale 1/sqrt(head_dim); query head h uses kv head
 * h / (num_heads / num_kv_heads) (contiguous GQA groups); a position
 * outside [0, max_len) is an error, the sequence is skipped and its output
 * rows are NaN.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared oracle.c -lm
 * (no fused multiply-add contraction, so x86 and Arm give identical bits).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARGS 1
#define ORACLE_ERR_NOMEM 2

/* ------------------------------------------------------------------------- */
/* KV scatter: the definition.                                               */
/*   for every sequence i and kv head g:                                     */
/*     cache[i][g][p_i][:] = rows[i][g][:]                                   */
/* Every other cache element is left untouched.  Returns the number of       */
/* sequences whose position was out of range (those are skipped).            */
/* ------------------------------------------------------------------------- */
int64_t oracle_kv_scatter(const float *k_rows, const float *v_rows,
                          const int32_t *positions, float *k_cache,
                          float *v_cache, int64_t M, int64_t num_kv_heads,
                          int64_t head_dim, int64_t max_len) {
  int64_t bad = 0;
  for (int64_t i = 0; i < M; ++i) {
    int64_t p = positions[i];
    if (p < 0 || p >= max_len) {
      ++bad;
      continue;
    }
    for (int64_t g = 0; g < num_kv_heads; ++g) {
      int64_t src = (i * num_kv_heads + g) * head_dim;
      int64_t dst = ((i * num_kv_heads + g) * max_len + p) * head_dim;
      memcpy(k_cache + dst, k_rows + src, (size_t)head_dim * sizeof(float));
      memcpy(v_cache + dst, v_rows + src, (size_t)head_dim * sizeof(float));
    }
  }
  return bad;
}

/* ------------------------------------------------------------------------- */
/* Softmax attention of one query row over L cache rows (the definition).    */
/* K and V are [L][D] with row stride D.  The result is left in double.      */
/* ------------------------------------------------------------------------- */
int oracle_attend_row_f64(const float *q, const float *K, const float *V,
                          int64_t L, int64_t D, double scale, double *out) {
  if (L < 1 || D < 1) return ORACLE_ERR_ARGS;
  double *s = (double *)malloc((size_t)L * sizeof(double));
  if (!s) return ORACLE_ERR_NOMEM;

  /* scores */
  for (int64_t j = 0; j < L; ++j) {
    double dot = 0.0;
    for (int64_t d = 0; d < D; ++d) dot += (double)q[d] * (double)K[j * D + d];
    s[j] = scale * dot;
  }
  /* running maximum of the scores */
  double m = s[0];
  for (int64_t j = 1; j < L; ++j)
    if (s[j] > m) m = s[j];
  /* weights and their sum */
  double Z = 0.0;
  for (int64_t j = 0; j < L; ++j) {
    s[j] = exp(s[j] - m);
    Z += s[j];
  }
  /* weighted mean of the value rows */
  for (int64_t d = 0; d < D; ++d) {
    double acc = 0.0;
    for (int64_t j = 0; j < L; ++j) acc += s[j] * (double)V[j * D + d];
    out[d] = acc / Z;
  }
  free(s);
  return ORACLE_OK;
}

/* f32 result: the double result rounded to nearest (C's default cast). */
int oracle_attend_row(const float *q, const float *K, const float *V,
                      int64_t L, int64_t D, double scale, float *out) {
  double *o = (double *)malloc((size_t)D * sizeof(double));
  if (!o) return ORACLE_ERR_NOMEM;
  int rc = oracle_attend_row_f64(q, K, V, L, D, scale, o);
  if (rc == ORACLE_OK)
    for (int64_t d = 0; d < D; ++d) out[d] = (float)o[d];
  free(o);
  return rc;
}

/* ------------------------------------------------------------------------- */
/* The split-K form (the pages' method): rows are cut into chunks of C rows; */
/* chunk c covers rows [cC, min((c+1)C, L)).  Each chunk yields its local    */
/* maximum m_c, local sum l_c = sum exp(s_j - m_c) and an unnormalised       */
/* accumulator acc_c[d] = sum exp(s_j - m_c) V[j][d].  The merge takes       */
/* M* = max_c m_c, rescales every partial by exp(m_c - M*) and divides.      */
/* Used only to pin the merge algebra against the definition above.          */
/* ------------------------------------------------------------------------- */
int oracle_attend_row_split_f64(const float *q, const float *K,
                                const float *V, int64_t L, int64_t D,
                                double scale, int64_t C, double *out) {
  if (L < 1 || D < 1 || C < 1) return ORACLE_ERR_ARGS;
  int64_t n = (L + C - 1) / C;
  double *pm = (double *)malloc((size_t)n * sizeof(double));
  double *pl = (double *)malloc((size_t)n * sizeof(double));
  double *pacc = (double *)malloc((size_t)(n * D) * sizeof(double));
  double *s = (double *)malloc((size_t)C * sizeof(double));
  if (!pm || !pl || !pacc || !s) {
    free(pm);
    free(pl);
    free(pacc);
    free(s);
    return ORACLE_ERR_NOMEM;
  }
  /* chunk partials */
  for (int64_t c = 0; c < n; ++c) {
    int64_t j0 = c * C;
    int64_t j1 = (j0 + C < L) ? j0 + C : L;
    for (int64_t j = j0; j < j1; ++j) {
      double dot = 0.0;
      for (int64_t d = 0; d < D; ++d)
        dot += (double)q[d] * (double)K[j * D + d];
      s[j - j0] = scale * dot;
    }
    double m = s[0];
    for (int64_t j = 1; j < j1 - j0; ++j)
      if (s[j] > m) m = s[j];
    double l = 0.0;
    for (int64_t j = 0; j < j1 - j0; ++j) {
      s[j] = exp(s[j] - m);
      l += s[j];
    }
    for (int64_t d = 0; d < D; ++d) {
      double a = 0.0;
      for (int64_t j = j0; j < j1; ++j) a += s[j - j0] * (double)V[j * D + d];
      pacc[c * D + d] = a;
    }
    pm[c] = m;
    pl[c] = l;
  }
  /* rescaling merge */
  double Ms = pm[0];
  for (int64_t c = 1; c < n; ++c)
    if (pm[c] > Ms) Ms = pm[c];
  double Z = 0.0;
  for (int64_t c = 0; c < n; ++c) Z += exp(pm[c] - Ms) * pl[c];
  for (int64_t d = 0; d < D; ++d) {
    double a = 0.0;
    for (int64_t c = 0; c < n; ++c) a += exp(pm[c] - Ms) * pacc[c * D + d];
    out[d] = a / Z;
  }
  free(pm);
  free(pl);
  free(pacc);
  free(s);
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* All query heads of one sequence.                                          */
/*   q   [H][D]                                                              */
/*   K,V [Hkv][row_stride][D]; rows 0..L-1 of each kv head are attended      */
/*   out [H][D]                                                              */
/* Query head h reads kv head h / (H / Hkv).                                 */
/* ------------------------------------------------------------------------- */
int oracle_attend_seq(const float *q, const float *K, const float *V,
                      int64_t L, int64_t row_stride, int64_t H, int64_t Hkv,
                      int64_t D, double scale, float *out) {
  if (H < 1 || Hkv < 1 || H % Hkv != 0 || L > row_stride) return ORACLE_ERR_ARGS;
  int64_t group = H / Hkv;
  for (int64_t h = 0; h < H; ++h) {
    int64_t g = h / group;
    const float *Kg = K + g * row_stride * D;
    const float *Vg = V + g * row_stride * D;
    int rc = oracle_attend_row(q + h * D, Kg, Vg, L, D, scale, out + h * D);
    if (rc != ORACLE_OK) return rc;
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* Whole decode attention over the cache layout [M][Hkv][max_len][D]         */
/* (after the scatter).  Sequence i attends rows 0..positions[i].  A         */
/* position outside [0, max_len) writes NaN to that sequence's output.      */
/* Returns the number of such sequences, or a negative error code.          */
/* ------------------------------------------------------------------------- */
int64_t oracle_decode(const float *q, const float *k_cache,
                      const float *v_cache, const int32_t *positions,
                      float *out, int64_t M, int64_t H, int64_t Hkv,
                      int64_t D, int64_t max_len) {
  double scale = 1.0 / sqrt((double)D);
  int64_t bad = 0;
  for (int64_t i = 0; i < M; ++i) {
    int64_t p = positions[i];
    float *o = out + i * H * D;
    if (p < 0 || p >= max_len) {
      for (int64_t e = 0; e < H * D; ++e) o[e] = NAN;
      ++bad;
      continue;
    }
    const float *Ki = k_cache + i * Hkv * max_len * D;
    const float *Vi = v_cache + i * Hkv * max_len * D;
    int rc = oracle_attend_seq(q + i * H * D, Ki, Vi, p + 1, max_len, H, Hkv,
                               D, scale, o);
    if (rc != ORACLE_OK) return -(int64_t)rc;
  }
  return bad;
}
