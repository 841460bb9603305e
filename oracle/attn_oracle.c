/*
 * Exact attention oracle: TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded fp64 restatement of what the attention hot
 * path computes.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load this file's library; the product path never does.
 * It shares no code, header or constant with the CUDA library.
 *
 * Definitions followed:
 *   - Forward, O = softmax(scale * Q K^T [+ causal mask]) V per head:
 *     SparkAttention (arXiv 2502.12784), Equation 1 and the masked decoder MHA
 *     of Figure 1; the same formula restated in the CANN ops-transformer MHA
 *     article, section 1 ("MHA 计算的瓦片化分解"), with scale = 1/sqrt(d_k).
 *   - Saved row statistic LSE_q = m_q + ln(sum_k exp(s_qk - m_q)):
 *     StreamKL summary (gist.science 2606.20005), Methodology 1 (LSE_t = m_t +
 *     log l_t) and 2 (probabilities regenerated as P = exp(S - LSE)).
 *   - Backward for the loss sum(O * dO): SparkAttention, Figure 9 / Equation 4
 *     (dPsum term, dS = P o (dP - dPsum)); the equation body is not printed on
 *     the page, so the exact gradient of the forward above is written out:
 *       dV = P^T dO,  dP = dO V^T,  D_q = sum_k P_qk dP_qk,
 *       dS = P o (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
 *
 * Conventions (the plainest readings where the pages are silent):
 *   - tensors are contiguous row-major [B][H][N][d]; LSE and D are [B][H][Nq];
 *   - causal = 1 is top-left aligned: query q sees keys k <= q;
 *   - causal = 2 is bottom-right aligned: the Nq queries are the last Nq
 *     positions of the Nk-long sequence (a decoder continuing a cached
 *     prefix; SparkAttention Figure 1, masked self-attention over preceding
 *     positions), so query q sees keys k <= q + Nk - Nq;
 *   - a query row that sees no key (bottom-right with Nq > Nk) has O = 0,
 *     LSE = -inf and zero gradients;
 *   - LSE is in natural-log units of the scaled scores;
 *   - D is the softmax Jacobian term sum_k P_qk dP_qk (mathematically equal to
 *     rowsum(dO o O)).
 *
 * No blocking, fusion or reordering beyond the definitions: each query row is
 * evaluated on its own from its full score row.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

/* Diagonal offset of the causal mask: query q sees keys k <= q + offset. */
static long mask_offset(int causal, long Nq, long Nk) { return causal == 2 ? Nk - Nq : 0; }

static int key_visible(long q, long k, int causal, long off) { return !causal || k <= q + off; }

static double dot(const double* a, const double* b, int d) {
  double acc = 0.0;
  for (int c = 0; c < d; ++c) acc += a[c] * b[c];
  return acc;
}

/*
 * Probabilities of one query row q of one head:
 *   s_k = scale <Q_q, K_k> for visible keys, m = max_k s_k,
 *   P_k = exp(s_k - m) / sum_j exp(s_j - m), masked keys get P_k = 0,
 *   *lse = m + ln(sum_j exp(s_j - m)).
 * Returns the number of visible keys (0 leaves P all zero and *lse = -inf).
 */
static long row_probs(const double* Qh, const double* Kh, long Nk, int d, long q,
                      int causal, long off, double scale, double* P, double* lse) {
  const double* qrow = Qh + (size_t)q * d;
  double m = -INFINITY;
  long nvis = 0;
  for (long k = 0; k < Nk; ++k) {
    if (key_visible(q, k, causal, off)) {
      P[k] = scale * dot(qrow, Kh + (size_t)k * d, d);
      if (P[k] > m) m = P[k];
      ++nvis;
    } else {
      P[k] = 0.0;
    }
  }
  if (nvis == 0) {
    *lse = -INFINITY;
    return 0;
  }
  double z = 0.0;
  for (long k = 0; k < Nk; ++k) {
    if (key_visible(q, k, causal, off)) {
      P[k] = exp(P[k] - m);
      z += P[k];
    }
  }
  for (long k = 0; k < Nk; ++k) P[k] /= z;
  *lse = m + log(z);
  return nvis;
}

/* dP_k = <dO_q, V_k> for every key; returns D_q = sum_k P_k dP_k. */
static double row_dp(const double* dOh, const double* Vh, long Nk, int d, long q,
                     const double* P, double* dP) {
  const double* dorow = dOh + (size_t)q * d;
  double D = 0.0;
  for (long k = 0; k < Nk; ++k) {
    dP[k] = dot(dorow, Vh + (size_t)k * d, d);
    D += P[k] * dP[k];
  }
  return D;
}

/* Full forward: O [B][H][Nq][d], LSE [B][H][Nq]. Returns 0, or -1 on allocation failure. */
int oracle_attn_fwd(const double* Q, const double* K, const double* V, double* O, double* LSE,
                    int B, int H, long Nq, long Nk, int d, int causal, double scale) {
  const long off = mask_offset(causal, Nq, Nk);
  double* P = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  if (!P) return -1;
  for (long bh = 0; bh < (long)B * H; ++bh) {
    const double* Qh = Q + (size_t)bh * Nq * d;
    const double* Kh = K + (size_t)bh * Nk * d;
    const double* Vh = V + (size_t)bh * Nk * d;
    for (long q = 0; q < Nq; ++q) {
      double lse;
      row_probs(Qh, Kh, Nk, d, q, causal, off, scale, P, &lse);
      double* orow = O + ((size_t)bh * Nq + q) * d;
      for (int c = 0; c < d; ++c) orow[c] = 0.0;
      for (long k = 0; k < Nk; ++k) {
        if (P[k] == 0.0) continue;
        const double* vrow = Vh + (size_t)k * d;
        for (int c = 0; c < d; ++c) orow[c] += P[k] * vrow[c];
      }
      LSE[(size_t)bh * Nq + q] = lse;
    }
  }
  free(P);
  return 0;
}

/*
 * Full backward of L = sum(O o dO): dQ [B][H][Nq][d], dK, dV [B][H][Nk][d];
 * Dout [B][H][Nq] (may be NULL) receives D_q = sum_k P_qk dP_qk.
 */
int oracle_attn_bwd(const double* Q, const double* K, const double* V, const double* dO,
                    double* dQ, double* dK, double* dV, double* Dout,
                    int B, int H, long Nq, long Nk, int d, int causal, double scale) {
  const long off = mask_offset(causal, Nq, Nk);
  double* P = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  double* dP = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  if (!P || !dP) {
    free(P);
    free(dP);
    return -1;
  }
  for (long bh = 0; bh < (long)B * H; ++bh) {
    const double* Qh = Q + (size_t)bh * Nq * d;
    const double* Kh = K + (size_t)bh * Nk * d;
    const double* Vh = V + (size_t)bh * Nk * d;
    const double* dOh = dO + (size_t)bh * Nq * d;
    double* dQh = dQ + (size_t)bh * Nq * d;
    double* dKh = dK + (size_t)bh * Nk * d;
    double* dVh = dV + (size_t)bh * Nk * d;
    memset(dKh, 0, sizeof(double) * (size_t)Nk * d);
    memset(dVh, 0, sizeof(double) * (size_t)Nk * d);
    for (long q = 0; q < Nq; ++q) {
      double lse;
      row_probs(Qh, Kh, Nk, d, q, causal, off, scale, P, &lse);
      double D = row_dp(dOh, Vh, Nk, d, q, P, dP);
      if (Dout) Dout[(size_t)bh * Nq + q] = D;
      double* dqrow = dQh + (size_t)q * d;
      const double* qrow = Qh + (size_t)q * d;
      const double* dorow = dOh + (size_t)q * d;
      for (int c = 0; c < d; ++c) dqrow[c] = 0.0;
      for (long k = 0; k < Nk; ++k) {
        if (!key_visible(q, k, causal, off)) continue;
        double dS = P[k] * (dP[k] - D);
        const double* krow = Kh + (size_t)k * d;
        double* dkrow = dKh + (size_t)k * d;
        double* dvrow = dVh + (size_t)k * d;
        for (int c = 0; c < d; ++c) {
          dqrow[c] += scale * dS * krow[c];
          dkrow[c] += scale * dS * qrow[c];
          dvrow[c] += P[k] * dorow[c];
        }
      }
    }
  }
  free(P);
  free(dP);
  return 0;
}

/*
 * Forward restricted to chosen query rows.  rows[i] = bh * Nq + q.
 * O_rows [nrows][d], lse_rows [nrows].  Same definition as oracle_attn_fwd.
 */
int oracle_attn_fwd_rows(const double* Q, const double* K, const double* V,
                         int B, int H, long Nq, long Nk, int d, int causal, double scale,
                         long nrows, const long* rows, double* O_rows, double* lse_rows) {
  const long off = mask_offset(causal, Nq, Nk);
  (void)B;
  (void)H;
  double* P = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  if (!P) return -1;
  for (long i = 0; i < nrows; ++i) {
    long bh = rows[i] / Nq, q = rows[i] % Nq;
    const double* Qh = Q + (size_t)bh * Nq * d;
    const double* Kh = K + (size_t)bh * Nk * d;
    const double* Vh = V + (size_t)bh * Nk * d;
    row_probs(Qh, Kh, Nk, d, q, causal, off, scale, P, &lse_rows[i]);
    double* orow = O_rows + (size_t)i * d;
    for (int c = 0; c < d; ++c) orow[c] = 0.0;
    for (long k = 0; k < Nk; ++k) {
      if (P[k] == 0.0) continue;
      for (int c = 0; c < d; ++c) orow[c] += P[k] * Vh[(size_t)k * d + c];
    }
  }
  free(P);
  return 0;
}

/* dQ restricted to chosen query rows (rows[i] = bh * Nq + q); dQ_rows [nrows][d], D_rows [nrows] (nullable). */
int oracle_attn_dq_rows(const double* Q, const double* K, const double* V, const double* dO,
                        int B, int H, long Nq, long Nk, int d, int causal, double scale,
                        long nrows, const long* rows, double* dQ_rows, double* D_rows) {
  const long off = mask_offset(causal, Nq, Nk);
  (void)B;
  (void)H;
  double* P = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  double* dP = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  if (!P || !dP) {
    free(P);
    free(dP);
    return -1;
  }
  for (long i = 0; i < nrows; ++i) {
    long bh = rows[i] / Nq, q = rows[i] % Nq;
    const double* Qh = Q + (size_t)bh * Nq * d;
    const double* Kh = K + (size_t)bh * Nk * d;
    const double* Vh = V + (size_t)bh * Nk * d;
    const double* dOh = dO + (size_t)bh * Nq * d;
    double lse;
    row_probs(Qh, Kh, Nk, d, q, causal, off, scale, P, &lse);
    double D = row_dp(dOh, Vh, Nk, d, q, P, dP);
    if (D_rows) D_rows[i] = D;
    double* dqrow = dQ_rows + (size_t)i * d;
    for (int c = 0; c < d; ++c) dqrow[c] = 0.0;
    for (long k = 0; k < Nk; ++k) {
      if (!key_visible(q, k, causal, off)) continue;
      double dS = P[k] * (dP[k] - D);
      for (int c = 0; c < d; ++c) dqrow[c] += scale * dS * Kh[(size_t)k * d + c];
    }
  }
  free(P);
  free(dP);
  return 0;
}

/*
 * The part of dK and dV of chosen key columns (cols[i] = bh * Nk + k) that
 * comes from the query rows q in [q_lo, q_hi): dK_k and dV_k are sums over
 * query rows, dK_k = scale sum_q dS_qk Q_q and dV_k = sum_q P_qk dO_q, and
 * this is that sum over the given rows only (the rows of any partition of
 * [0, Nq) add up to the whole).  dK_cols, dV_cols [ncols][d].  Every query
 * row taken is evaluated in full (its whole score row), exactly as in
 * oracle_attn_bwd.
 */
int oracle_attn_dkdv_cols_part(const double* Q, const double* K, const double* V, const double* dO,
                               int B, int H, long Nq, long Nk, int d, int causal, double scale,
                               long ncols, const long* cols, long q_lo, long q_hi,
                               double* dK_cols, double* dV_cols) {
  const long off = mask_offset(causal, Nq, Nk);
  if (q_lo < 0) q_lo = 0;
  if (q_hi > Nq) q_hi = Nq;
  double* P = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  double* dP = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  if (!P || !dP) {
    free(P);
    free(dP);
    return -1;
  }
  memset(dK_cols, 0, sizeof(double) * (size_t)ncols * d);
  memset(dV_cols, 0, sizeof(double) * (size_t)ncols * d);
  for (long bh = 0; bh < (long)B * H; ++bh) {
    /* smallest chosen key of this head: rows q < kmin - off see none of them when causal */
    long kmin = -1;
    for (long i = 0; i < ncols; ++i)
      if (cols[i] / Nk == bh && (kmin < 0 || cols[i] % Nk < kmin)) kmin = cols[i] % Nk;
    if (kmin < 0) continue;
    const double* Qh = Q + (size_t)bh * Nq * d;
    const double* Kh = K + (size_t)bh * Nk * d;
    const double* Vh = V + (size_t)bh * Nk * d;
    const double* dOh = dO + (size_t)bh * Nq * d;
    long q0 = (causal && kmin - off > 0) ? kmin - off : 0;
    if (q0 < q_lo) q0 = q_lo;
    for (long q = q0; q < q_hi; ++q) {
      double lse;
      row_probs(Qh, Kh, Nk, d, q, causal, off, scale, P, &lse);
      double D = row_dp(dOh, Vh, Nk, d, q, P, dP);
      const double* qrow = Qh + (size_t)q * d;
      const double* dorow = dOh + (size_t)q * d;
      for (long i = 0; i < ncols; ++i) {
        if (cols[i] / Nk != bh) continue;
        long k = cols[i] % Nk;
        if (!key_visible(q, k, causal, off)) continue;
        double dS = P[k] * (dP[k] - D);
        for (int c = 0; c < d; ++c) {
          dK_cols[(size_t)i * d + c] += scale * dS * qrow[c];
          dV_cols[(size_t)i * d + c] += P[k] * dorow[c];
        }
      }
    }
  }
  free(P);
  free(dP);
  return 0;
}

/* dK and dV of chosen key columns (cols[i] = bh * Nk + k) over all query rows. */
int oracle_attn_dkdv_cols(const double* Q, const double* K, const double* V, const double* dO,
                          int B, int H, long Nq, long Nk, int d, int causal, double scale,
                          long ncols, const long* cols, double* dK_cols, double* dV_cols) {
  return oracle_attn_dkdv_cols_part(Q, K, V, dO, B, H, Nq, Nk, d, causal, scale, ncols, cols, 0, Nq, dK_cols,
                                    dV_cols);
}

/* The full probability matrix of one head, P [Nq][Nk] (small shapes; used by invariant checks). */
int oracle_attn_probs(const double* Qh, const double* Kh, long Nq, long Nk, int d, int causal,
                      double scale, double* P, double* lse) {
  const long off = mask_offset(causal, Nq, Nk);
  for (long q = 0; q < Nq; ++q) row_probs(Qh, Kh, Nk, d, q, causal, off, scale, P + (size_t)q * Nk, &lse[q]);
  return 0;
}

/* ------------------------------------------------------------------------
 * Attention KL divergence (StreamKL summary, gist.science 2606.20005).
 *
 * Two attention distributions over the same keys positions, a teacher (1) and
 * a student (2), each from its own queries and keys:
 *   S_t = scale Q_t K_t^T (visible keys only), P_t = softmax_row(S_t),
 *   LSE_t = m_t + ln sum_k exp(S_t - m_t)                  (Methodology 1)
 * and the row-wise divergence of the student from the teacher
 *   KL_q = sum_k P1_qk (log P1_qk - log P2_qk),  log P_t = S_t - LSE_t.
 * Gradients of L = sum_q g_q KL_q (Methodology 2, P regenerated from LSE):
 *   setting 1 (teacher fixed, the student is trained):
 *     dS2_qk = g_q (P2_qk - P1_qk)
 *   setting 2 (student fixed, the teacher is trained):
 *     dS1_qk = g_q P1_qk ((S1_qk - LSE1_q) - (S2_qk - LSE2_q) - KL_q)
 *   then dQ_t = scale dS_t K_t and dK_t = scale dS_t^T Q_t for the trained
 *   distribution t.  The masks are those of the attention oracle above; a row
 *   that sees no key has KL = 0, LSE_t = -inf and zero gradients.
 * ------------------------------------------------------------------------ */

/* Both distributions of one row; returns the number of visible keys. */
static long kl_row(const double* Q1h, const double* K1h, const double* Q2h, const double* K2h, long Nk, int d,
                   long q, int causal, long off, double scale, double* P1, double* P2, double* lse1, double* lse2,
                   double* kl) {
  long n = row_probs(Q1h, K1h, Nk, d, q, causal, off, scale, P1, lse1);
  row_probs(Q2h, K2h, Nk, d, q, causal, off, scale, P2, lse2);
  double acc = 0.0;
  for (long k = 0; k < Nk && n > 0; ++k) {
    if (!key_visible(q, k, causal, off) || P1[k] == 0.0) continue;
    const double s1 = scale * dot(Q1h + (size_t)q * d, K1h + (size_t)k * d, d);
    const double s2 = scale * dot(Q2h + (size_t)q * d, K2h + (size_t)k * d, d);
    acc += P1[k] * ((s1 - *lse1) - (s2 - *lse2));
  }
  *kl = n > 0 ? acc : 0.0;
  return n;
}

/* KL, LSE1, LSE2 [B][H][Nq]. */
int oracle_kl_fwd(const double* Q1, const double* K1, const double* Q2, const double* K2, double* KL, double* LSE1,
                  double* LSE2, int B, int H, long Nq, long Nk, int d, int causal, double scale) {
  const long off = mask_offset(causal, Nq, Nk);
  double* P1 = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  double* P2 = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  if (!P1 || !P2) {
    free(P1);
    free(P2);
    return -1;
  }
  for (long bh = 0; bh < (long)B * H; ++bh) {
    const size_t qo = (size_t)bh * Nq * d, ko = (size_t)bh * Nk * d;
    for (long q = 0; q < Nq; ++q) {
      const size_t r = (size_t)bh * Nq + q;
      kl_row(Q1 + qo, K1 + ko, Q2 + qo, K2 + ko, Nk, d, q, causal, off, scale, P1, P2, &LSE1[r], &LSE2[r], &KL[r]);
    }
  }
  free(P1);
  free(P2);
  return 0;
}

/* dS of one row for the trained distribution (setting 1: student, 2: teacher); dS [Nk]. */
static void kl_row_ds(const double* Q1h, const double* K1h, const double* Q2h, const double* K2h, long Nk, int d,
                      long q, int causal, long off, double scale, double g, int setting, double* P1, double* P2,
                      double* dS) {
  double lse1, lse2, kl;
  long n = kl_row(Q1h, K1h, Q2h, K2h, Nk, d, q, causal, off, scale, P1, P2, &lse1, &lse2, &kl);
  for (long k = 0; k < Nk; ++k) {
    dS[k] = 0.0;
    if (n == 0 || !key_visible(q, k, causal, off)) continue;
    if (setting == 1) {
      dS[k] = g * (P2[k] - P1[k]);
    } else {
      const double s1 = scale * dot(Q1h + (size_t)q * d, K1h + (size_t)k * d, d);
      const double s2 = scale * dot(Q2h + (size_t)q * d, K2h + (size_t)k * d, d);
      dS[k] = g * P1[k] * ((s1 - lse1) - (s2 - lse2) - kl);
    }
  }
}

/*
 * Gradients of sum_q G_q KL_q for the trained distribution: dQ [B][H][Nq][d] and dK [B][H][Nk][d] of the
 * student (setting 1) or of the teacher (setting 2).  G [B][H][Nq].
 */
int oracle_kl_bwd(const double* Q1, const double* K1, const double* Q2, const double* K2, const double* G,
                  int setting, double* dQ, double* dK, int B, int H, long Nq, long Nk, int d, int causal,
                  double scale) {
  if (setting != 1 && setting != 2) return -2;
  const long off = mask_offset(causal, Nq, Nk);
  double* P1 = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  double* P2 = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  double* dS = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  if (!P1 || !P2 || !dS) {
    free(P1);
    free(P2);
    free(dS);
    return -1;
  }
  for (long bh = 0; bh < (long)B * H; ++bh) {
    const size_t qo = (size_t)bh * Nq * d, ko = (size_t)bh * Nk * d;
    const double* Qt = (setting == 1 ? Q2 : Q1) + qo;
    const double* Kt = (setting == 1 ? K2 : K1) + ko;
    double* dKh = dK + ko;
    memset(dKh, 0, sizeof(double) * (size_t)Nk * d);
    for (long q = 0; q < Nq; ++q) {
      kl_row_ds(Q1 + qo, K1 + ko, Q2 + qo, K2 + ko, Nk, d, q, causal, off, scale, G[(size_t)bh * Nq + q], setting,
                P1, P2, dS);
      double* dqrow = dQ + qo + (size_t)q * d;
      for (int c = 0; c < d; ++c) dqrow[c] = 0.0;
      for (long k = 0; k < Nk; ++k) {
        if (dS[k] == 0.0) continue;
        for (int c = 0; c < d; ++c) {
          dqrow[c] += scale * dS[k] * Kt[(size_t)k * d + c];
          dKh[(size_t)k * d + c] += scale * dS[k] * Qt[(size_t)q * d + c];
        }
      }
    }
  }
  free(P1);
  free(P2);
  free(dS);
  return 0;
}

/* KL, LSE1, LSE2 of chosen rows (rows[i] = bh * Nq + q). */
int oracle_kl_fwd_rows(const double* Q1, const double* K1, const double* Q2, const double* K2, int B, int H, long Nq,
                       long Nk, int d, int causal, double scale, long nrows, const long* rows, double* KL,
                       double* LSE1, double* LSE2) {
  (void)B;
  (void)H;
  const long off = mask_offset(causal, Nq, Nk);
  double* P1 = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  double* P2 = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  if (!P1 || !P2) {
    free(P1);
    free(P2);
    return -1;
  }
  for (long i = 0; i < nrows; ++i) {
    const long bh = rows[i] / Nq, q = rows[i] % Nq;
    const size_t qo = (size_t)bh * Nq * d, ko = (size_t)bh * Nk * d;
    kl_row(Q1 + qo, K1 + ko, Q2 + qo, K2 + ko, Nk, d, q, causal, off, scale, P1, P2, &LSE1[i], &LSE2[i], &KL[i]);
  }
  free(P1);
  free(P2);
  return 0;
}

/* dQ of the trained distribution for chosen rows (rows[i] = bh * Nq + q); dQ_rows [nrows][d]. */
int oracle_kl_dq_rows(const double* Q1, const double* K1, const double* Q2, const double* K2, const double* G,
                      int setting, int B, int H, long Nq, long Nk, int d, int causal, double scale, long nrows,
                      const long* rows, double* dQ_rows) {
  (void)B;
  (void)H;
  if (setting != 1 && setting != 2) return -2;
  const long off = mask_offset(causal, Nq, Nk);
  double* P1 = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  double* P2 = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  double* dS = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  if (!P1 || !P2 || !dS) {
    free(P1);
    free(P2);
    free(dS);
    return -1;
  }
  for (long i = 0; i < nrows; ++i) {
    const long bh = rows[i] / Nq, q = rows[i] % Nq;
    const size_t qo = (size_t)bh * Nq * d, ko = (size_t)bh * Nk * d;
    const double* Kt = (setting == 1 ? K2 : K1) + ko;
    kl_row_ds(Q1 + qo, K1 + ko, Q2 + qo, K2 + ko, Nk, d, q, causal, off, scale, G[(size_t)bh * Nq + q], setting,
              P1, P2, dS);
    double* dqrow = dQ_rows + (size_t)i * d;
    for (int c = 0; c < d; ++c) dqrow[c] = 0.0;
    for (long k = 0; k < Nk; ++k) {
      if (dS[k] == 0.0) continue;
      for (int c = 0; c < d; ++c) dqrow[c] += scale * dS[k] * Kt[(size_t)k * d + c];
    }
  }
  free(P1);
  free(P2);
  free(dS);
  return 0;
}

/*
 * The part of dK of the trained distribution, for chosen key rows (cols[i] =
 * bh * Nk + k), that comes from the query rows q in [q_lo, q_hi): dK_k =
 * scale sum_q dS_qk Q_q summed over the given rows only (the rows of any
 * partition of [0, Nq) add up to the whole).  dK_cols [ncols][d].
 */
int oracle_kl_dk_cols_part(const double* Q1, const double* K1, const double* Q2, const double* K2, const double* G,
                           int setting, int B, int H, long Nq, long Nk, int d, int causal, double scale, long ncols,
                           const long* cols, long q_lo, long q_hi, double* dK_cols) {
  if (setting != 1 && setting != 2) return -2;
  const long off = mask_offset(causal, Nq, Nk);
  if (q_lo < 0) q_lo = 0;
  if (q_hi > Nq) q_hi = Nq;
  double* P1 = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  double* P2 = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  double* dS = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  if (!P1 || !P2 || !dS) {
    free(P1);
    free(P2);
    free(dS);
    return -1;
  }
  memset(dK_cols, 0, sizeof(double) * (size_t)ncols * d);
  for (long bh = 0; bh < (long)B * H; ++bh) {
    long kmin = -1;
    for (long i = 0; i < ncols; ++i)
      if (cols[i] / Nk == bh && (kmin < 0 || cols[i] % Nk < kmin)) kmin = cols[i] % Nk;
    if (kmin < 0) continue;
    const size_t qo = (size_t)bh * Nq * d, ko = (size_t)bh * Nk * d;
    const double* Qt = (setting == 1 ? Q2 : Q1) + qo;
    long q0 = (causal && kmin - off > 0) ? kmin - off : 0;
    if (q0 < q_lo) q0 = q_lo;
    for (long q = q0; q < q_hi; ++q) {
      kl_row_ds(Q1 + qo, K1 + ko, Q2 + qo, K2 + ko, Nk, d, q, causal, off, scale, G[(size_t)bh * Nq + q], setting,
                P1, P2, dS);
      for (long i = 0; i < ncols; ++i) {
        if (cols[i] / Nk != bh) continue;
        const long k = cols[i] % Nk;
        if (dS[k] == 0.0) continue;
        for (int c = 0; c < d; ++c) dK_cols[(size_t)i * d + c] += scale * dS[k] * Qt[(size_t)q * d + c];
      }
    }
  }
  free(P1);
  free(P2);
  free(dS);
  return 0;
}

/* dK of the trained distribution for chosen key rows (cols[i] = bh * Nk + k) over all query rows. */
int oracle_kl_dk_cols(const double* Q1, const double* K1, const double* Q2, const double* K2, const double* G,
                      int setting, int B, int H, long Nq, long Nk, int d, int causal, double scale, long ncols,
                      const long* cols, double* dK_cols) {
  return oracle_kl_dk_cols_part(Q1, K1, Q2, K2, G, setting, B, H, Nq, Nk, d, causal, scale, ncols, cols, 0, Nq,
                                dK_cols);
}
