/*
 * Oracle for the DiT blockwise-attention path -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, fp64 CPU restatement of what the GPU path computes. Only the
 * tests, the smoke check and the benchmark's CPU-baseline leg may load it; the
 * product library never links, loads or calls it, and this file shares no
 * code, header or constant with the CUDA sources.
 *
 * What is computed, and where it comes from:
 *  - Full bidirectional softmax attention over a DiT token sequence (image
 *    latent patches, plus text tokens for joint attention).  The xDiT page
 *    ("xDiT: an Inference Engine for DiTs with Massive Parallelism", abstract)
 *    names attention over the token sequence as the cost that grows with the
 *    sequence length and that sequence parallelism splits.  The pages print no
 *    formula; the plainest reading is the textbook scaled dot-product
 *    attention, per (batch, head):
 *        score_ij = (q_i . k_j) / sqrt(D)
 *        LSE_i    = m_i + ln sum_j exp(score_ij - m_i),  m_i = max_j score_ij
 *        O_i      = sum_j exp(score_ij - LSE_i) v_j
 *  - Attention restricted to a contiguous key range [j0, j1): the per-device
 *    (per-chunk) computation of ring / Torus attention, where each device sees
 *    one piece of K/V at a time ("SwiftFusion: Scalable Sequence Parallelism
 *    ...", ideas 1 and 2: ring attention, Torus attention computing each
 *    received piece as it arrives).
 *  - The merge of per-chunk partial results (O_c, LSE_c) by log-sum-exp
 *    weights, the reduction that recombines the pieces of that split:
 *        M = max_c LSE_c,  LSE = M + ln sum_c exp(LSE_c - M),
 *        O = sum_c exp(LSE_c - LSE) O_c
 *    Chunks with LSE_c = -inf carry weight zero and their O_c is not read.
 *  - The classifier-free-guidance combine of the conditional and the
 *    unconditional noise predictions ("Accelerating Diffusion via Hybrid
 *    Data-Pipeline Parallelism Based on Conditional Guidance Scheduling",
 *    Technische Zusammenfassung 2A: the path with prompt c and the path with
 *    c = empty), in its standard form out = eps_u + w (eps_c - eps_u).
 *  - The discrepancy between the two paths that the same page (section 2B,
 *    adaptive parallelism switching) measures to pick its phase switch points,
 *    named rel-MAE there without a formula.  Plainest reading: the mean
 *    absolute difference relative to the mean absolute unconditional noise,
 *        rel-MAE = sum_i |eps_c[i] - eps_u[i]| / sum_i |eps_u[i]|,
 *    computed in the same pass as the combine.  The two sums and their ratio
 *    are returned.  The page does not say what happens when the unconditional
 *    noise is all zero; the reading taken is the limit of identical paths:
 *    0 when the difference sum is 0 too, +inf otherwise.
 *
 * Layouts: q, k, v, out are [BH][S][D] row-major doubles; lse is [BH][S].
 * Every loop is the definition written out, with no blocking or reordering.
 */
#include <math.h>
#include <omp.h>
#include <stddef.h>
#include <stdlib.h>

/* One query row against keys [j0, j1) of one (batch, head).  Writes D values
 * to out_row and the natural-log LSE to *lse_row.  scores is caller scratch of
 * length j1 - j0. */
static void attn_one_row(const double *q_row, const double *k_bh,
                         const double *v_bh, long long j0, long long j1, int D,
                         double *scores, double *out_row, double *lse_row) {
  const double scale = 1.0 / sqrt((double)D);
  double m = -INFINITY;
  for (long long j = j0; j < j1; ++j) {
    const double *k_row = k_bh + j * (long long)D;
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += q_row[d] * k_row[d];
    double s = dot * scale;
    scores[j - j0] = s;
    if (s > m) m = s;
  }
  double z = 0.0;
  for (long long j = j0; j < j1; ++j) z += exp(scores[j - j0] - m);
  const double lse = m + log(z);
  for (int d = 0; d < D; ++d) out_row[d] = 0.0;
  for (long long j = j0; j < j1; ++j) {
    const double p = exp(scores[j - j0] - lse);
    const double *v_row = v_bh + j * (long long)D;
    for (int d = 0; d < D; ++d) out_row[d] += p * v_row[d];
  }
  *lse_row = lse;
}

/* Attention of every query row of every (batch, head) over keys [j0, j1).
 * Returns 0, or -1 on an empty or out-of-range key range. */
int oracle_attn_range(const double *q, const double *k, const double *v,
                      long long BH, long long S, int D, long long j0,
                      long long j1, double *out, double *lse) {
  if (j0 < 0 || j1 > S || j0 >= j1 || D < 1) return -1;
  const long long total = BH * S;
#pragma omp parallel for schedule(dynamic, 16)
  for (long long r = 0; r < total; ++r) {
    const long long bh = r / S;
    double *scores = (double *)malloc(sizeof(double) * (size_t)(j1 - j0));
    attn_one_row(q + r * (long long)D, k + bh * S * (long long)D,
                 v + bh * S * (long long)D, j0, j1, D, scores,
                 out + r * (long long)D, lse + r);
    free(scores);
  }
  return 0;
}

/* Attention for a list of sampled rows: rows[t] = bh * S + i.  Writes
 * out[t][D] and lse[t].  Used to check full-size outputs one row at a time. */
int oracle_attn_rows(const double *q, const double *k, const double *v,
                     long long BH, long long S, int D, const long long *rows,
                     long long nrows, long long j0, long long j1, double *out,
                     double *lse) {
  if (j0 < 0 || j1 > S || j0 >= j1 || D < 1) return -1;
  for (long long t = 0; t < nrows; ++t)
    if (rows[t] < 0 || rows[t] >= BH * S) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (long long t = 0; t < nrows; ++t) {
    const long long r = rows[t];
    const long long bh = r / S;
    double *scores = (double *)malloc(sizeof(double) * (size_t)(j1 - j0));
    attn_one_row(q + r * (long long)D, k + bh * S * (long long)D,
                 v + bh * S * (long long)D, j0, j1, D, scores,
                 out + t * (long long)D, lse + t);
    free(scores);
  }
  return 0;
}

/* Log-sum-exp merge of n partial results.  partials is [n][rows][D], lses is
 * [n][rows]; out is [rows][D], lse_out is [rows] (may be NULL).  A row whose
 * partial LSEs are all -inf gets out = 0 and lse = -inf. */
int oracle_lse_merge(const double *partials, const double *lses, int n,
                     long long rows, int D, double *out, double *lse_out) {
  if (n < 1 || rows < 0 || D < 1) return -1;
#pragma omp parallel for schedule(static)
  for (long long r = 0; r < rows; ++r) {
    double m = -INFINITY;
    for (int c = 0; c < n; ++c) {
      const double l = lses[(long long)c * rows + r];
      if (l > m) m = l;
    }
    double *o = out + r * (long long)D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (m == -INFINITY) {
      if (lse_out) lse_out[r] = -INFINITY;
      continue;
    }
    double z = 0.0;
    for (int c = 0; c < n; ++c) {
      const double l = lses[(long long)c * rows + r];
      if (l == -INFINITY) continue;
      z += exp(l - m);
    }
    const double lse = m + log(z);
    for (int c = 0; c < n; ++c) {
      const double l = lses[(long long)c * rows + r];
      if (l == -INFINITY) continue;
      const double wgt = exp(l - lse);
      const double *oc = partials + ((long long)c * rows + r) * (long long)D;
      for (int d = 0; d < D; ++d) o[d] += wgt * oc[d];
    }
    if (lse_out) lse_out[r] = lse;
  }
  return 0;
}

/* Classifier-free guidance combine, elementwise. */
int oracle_cfg_combine(const double *eps_c, const double *eps_u, double w,
                       double *out, long long numel) {
  if (numel < 0) return -1;
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < numel; ++i)
    out[i] = eps_u[i] + w * (eps_c[i] - eps_u[i]);
  return 0;
}

/* Classifier-free guidance combine plus the rel-MAE discrepancy:
 * sums[0] = sum |eps_c - eps_u|, sums[1] = sum |eps_u|,
 * sums[2] = sums[0] / sums[1] (0 if both are 0, +inf if only sums[1] is). */
int oracle_cfg_relmae(const double *eps_c, const double *eps_u, double w,
                      double *out, long long numel, double *sums) {
  if (numel < 0) return -1;
  double diff = 0.0, base = 0.0;
  for (long long i = 0; i < numel; ++i) {
    const double d = eps_c[i] - eps_u[i];
    out[i] = eps_u[i] + w * d;
    diff += fabs(d);
    base += fabs(eps_u[i]);
  }
  sums[0] = diff;
  sums[1] = base;
  if (base > 0.0)
    sums[2] = diff / base;
  else
    sums[2] = diff == 0.0 ? 0.0 : INFINITY;
  return 0;
}

/* Number of OpenMP threads the loops above run on (for reporting). */
int oracle_num_threads(void) {
  int n = 1;
#pragma omp parallel
  {
#pragma omp single
    n = omp_get_num_threads();
  }
  return n;
}
