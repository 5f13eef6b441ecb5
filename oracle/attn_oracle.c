/*
 * attn_oracle.c -- the fp64 CPU oracle for the fused attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the test suite, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * What it computes (the plain definition, no tiling, no online softmax):
 *   for one (batch, head) slice and one query row i,
 *     s_j   = scale * sum_d q_{i,d} k_{j,d}        for every visible key j
 *     m     = max_j s_j
 *     LSE_i = m + ln( sum_j exp(s_j - m) )
 *     P_ij  = exp(s_j - LSE_i)
 *     O_i,d = sum_j P_ij v_{j,d}
 *   Visible keys: all j < N, or j <= i under the causal mask.
 *
 * Sources:
 *   - The attention definition O = softmax(Q K^T * scale) V that both kernel
 *     examples compute: ThunderKittens news write-up (88811315.cn, post
 *     77732), "RTX 4090 flash attention" example and "H100 FlashAttention-2
 *     forward" example; the same kernels in the GeekNews summary
 *     (es.news.hada.io topic 14783), section "Ejemplo de FlashAttention y
 *     rendimiento".  The examples scale scores by 1/sqrt(64) = 0.125 and
 *     1/sqrt(128) ~= 0.08838834764; here the scale is an argument.
 *   - The causal mask (key j visible to query i iff j <= i, diagonal
 *     included) and the per-row log-sum-exp are not on those pages; they are
 *     the plainest reading of the requested interface: natural log of the sum
 *     of exp over the scaled, masked scores.
 *
 * Precision: every bf16 input is widened exactly to double; all arithmetic is
 * IEEE double in plain loop order.  The score row is materialised in full
 * (N doubles per thread), so memory stays O(N) per thread.
 *
 * Inputs are bf16 bit patterns (uint16), layout [BH, N, D] row-major
 * (BH = batch * heads).  Rows are addressed by their flat index bh*N + i.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact bf16 -> double widening: a bf16 value is the high half of a float. */
static double widen_bf16(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/*
 * One query row.  `scores` is caller-provided scratch of N doubles.
 * `shift` is added to every score of the row before the softmax; it exists so
 * tests can check that a per-row constant leaves O unchanged and moves LSE by
 * exactly that constant.  Pass 0.0 for the plain definition.
 */
static void one_row(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    int64_t N, int64_t D, double scale, int causal,
                    int64_t bh, int64_t i, double shift, double *scores,
                    double *o_row, double *lse_out) {
  const uint16_t *qi = q + (bh * N + i) * D;
  const uint16_t *kb = k + bh * N * D;
  const uint16_t *vb = v + bh * N * D;
  int64_t nvis = causal ? (i + 1) : N;

  /* s_j = scale * q_i . k_j (+ shift) */
  double m = -INFINITY;
  for (int64_t j = 0; j < nvis; ++j) {
    const uint16_t *kj = kb + j * D;
    double dot = 0.0;
    for (int64_t d = 0; d < D; ++d) dot += widen_bf16(qi[d]) * widen_bf16(kj[d]);
    double s = scale * dot + shift;
    scores[j] = s;
    if (s > m) m = s;
  }

  /* LSE = m + ln sum_j exp(s_j - m) */
  double z = 0.0;
  for (int64_t j = 0; j < nvis; ++j) z += exp(scores[j] - m);
  double lse = m + log(z);

  /* P_j = exp(s_j - LSE); O = sum_j P_j v_j */
  for (int64_t d = 0; d < D; ++d) o_row[d] = 0.0;
  for (int64_t j = 0; j < nvis; ++j) {
    double p = exp(scores[j] - lse);
    const uint16_t *vj = vb + j * D;
    for (int64_t d = 0; d < D; ++d) o_row[d] += p * widen_bf16(vj[d]);
  }
  *lse_out = lse;
}

/*
 * attn_oracle_rows: compute O and LSE for a list of rows.
 *
 *   q, k, v   bf16 bits, [BH, N, D] row-major
 *   rows      flat row indices bh*N + i (NULL = every row, in order)
 *   nrows     number of entries in `rows` (ignored when rows == NULL)
 *   shifts    per-requested-row additive score shift (NULL = none)
 *   o         out: [nrows, D] doubles   (or [BH*N, D] when rows == NULL)
 *   lse       out: [nrows] doubles
 *   nthreads  OpenMP threads to use (<= 0: library default)
 *
 * Returns the number of threads used, or -1 on a bad argument.
 */
int attn_oracle_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     int64_t BH, int64_t N, int64_t D, double scale, int causal,
                     const int64_t *rows, int64_t nrows, const double *shifts,
                     double *o, double *lse, int nthreads) {
  if (!q || !k || !v || !o || !lse || BH <= 0 || N <= 0 || D <= 0) return -1;
  int64_t total = rows ? nrows : BH * N;
  if (total < 0) return -1;
  if (rows) {
    for (int64_t r = 0; r < nrows; ++r)
      if (rows[r] < 0 || rows[r] >= BH * N) return -1;
  }
  int used = 1;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
  {
#pragma omp single
    used = omp_get_num_threads();
  }
#else
  (void)nthreads;
#endif
  int failed = 0;
#pragma omp parallel
  {
    double *scores = (double *)malloc((size_t)N * sizeof(double));
    if (!scores) {
#pragma omp atomic write
      failed = 1;
    }
    /* every thread reaches the work-sharing loop, even one whose buffer failed */
#pragma omp for schedule(dynamic, 4)
    for (int64_t r = 0; r < total; ++r) {
      if (!scores) continue;
      int64_t flat = rows ? rows[r] : r;
      int64_t bh = flat / N, i = flat % N;
      double sh = shifts ? shifts[r] : 0.0;
      one_row(q, k, v, N, D, scale, causal, bh, i, sh, scores, o + r * D, lse + r);
    }
    free(scores);
  }
  return failed ? -1 : used;
}

/*
 * Queries and keys of different lengths (Nq query rows, Nk keys per slice),
 * the shape of attention at inference time: a block of new queries against
 * a longer run of cached keys.  Same definition as above, with the visible
 * keys of query i being all j < Nk, or, under the causal mask aligned to
 * the end of the key sequence, j <= i + (Nk - Nq) (query i is the
 * (Nk - Nq + i)-th position of the sequence).  For Nq == Nk this is the mask
 * above.  Neither page fixes the alignment for Nq != Nk; this is the reading
 * where the queries are the last Nq positions of the sequence.
 *
 *   q  bf16 bits [BH, Nq, D];  k, v  bf16 bits [BH, Nk, D]
 *   rows      flat query-row indices bh*Nq + i (NULL = every row, in order)
 *   o, lse    out: [nrows, D] and [nrows] doubles
 * Returns the number of threads used, or -1 on a bad argument (including a
 * causal Nq > Nk, where the first queries would see no key).
 */
static void one_row_qk(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       int64_t Nq, int64_t Nk, int64_t D, double scale, int causal,
                       int64_t bh, int64_t i, double *scores, double *o_row, double *lse_out) {
  const uint16_t *qi = q + (bh * Nq + i) * D;
  const uint16_t *kb = k + bh * Nk * D;
  const uint16_t *vb = v + bh * Nk * D;
  const int64_t nvis = causal ? (i + (Nk - Nq) + 1) : Nk;
  double m = -INFINITY;
  for (int64_t j = 0; j < nvis; ++j) {
    const uint16_t *kj = kb + j * D;
    double dot = 0.0;
    for (int64_t d = 0; d < D; ++d) dot += widen_bf16(qi[d]) * widen_bf16(kj[d]);
    double s = scale * dot;
    scores[j] = s;
    if (s > m) m = s;
  }
  double z = 0.0;
  for (int64_t j = 0; j < nvis; ++j) z += exp(scores[j] - m);
  double lse = m + log(z);
  for (int64_t d = 0; d < D; ++d) o_row[d] = 0.0;
  for (int64_t j = 0; j < nvis; ++j) {
    double p = exp(scores[j] - lse);
    const uint16_t *vj = vb + j * D;
    for (int64_t d = 0; d < D; ++d) o_row[d] += p * widen_bf16(vj[d]);
  }
  *lse_out = lse;
}

int attn_oracle_rows_qk(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t BH,
                        int64_t Nq, int64_t Nk, int64_t D, double scale, int causal,
                        const int64_t *rows, int64_t nrows, double *o, double *lse,
                        int nthreads) {
  if (!q || !k || !v || !o || !lse || BH <= 0 || Nq <= 0 || Nk <= 0 || D <= 0) return -1;
  if (causal && Nq > Nk) return -1;
  int64_t total = rows ? nrows : BH * Nq;
  if (total < 0) return -1;
  if (rows) {
    for (int64_t r = 0; r < nrows; ++r)
      if (rows[r] < 0 || rows[r] >= BH * Nq) return -1;
  }
  int used = 1;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
  {
#pragma omp single
    used = omp_get_num_threads();
  }
#else
  (void)nthreads;
#endif
  int failed = 0;
#pragma omp parallel
  {
    double *scores = (double *)malloc((size_t)Nk * sizeof(double));
    if (!scores) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 4)
    for (int64_t r = 0; r < total; ++r) {
      if (!scores) continue;
      int64_t flat = rows ? rows[r] : r;
      one_row_qk(q, k, v, Nq, Nk, D, scale, causal, flat / Nq, flat % Nq, scores, o + r * D,
                 lse + r);
    }
    free(scores);
  }
  return failed ? -1 : used;
}

/* Threads an OpenMP region would use by default (for reporting). */
int attn_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
