/*
 * Row scalars of the exact attention backward-over-backward, in plain C and
 * fp64, for sequences too long for the numpy oracle to finish in seconds.
 *
 * TEST INFRASTRUCTURE ONLY (part of the oracle): called by the tests through
 * oracle/crows.py; the CUDA library never links or calls it, and it shares no
 * code with the CUDA path.
 *
 * For every query row i of one (batch, head), with tau the score scale:
 *   S_ij = tau Q_i.K_j (keys j > i masked when causal),
 *   L_i  = log sum_j exp(S_ij)                     [FAB] section 二
 *   P_ij = exp(S_ij - L_i),  O_i = sum_j P_ij V_j,  D_i = dO_i.O_i
 *   F_ij = tau (U_Q,i.K_j + Q_i.U_K,j),  alpha_i = sum_j P_ij F_ij
 *   dP_ij = dO_i.V_j,  G_ij = dO_i.U_V,j,
 *   E_i  = sum_j P_ij (F_ij (dP_ij - D_i) + G_ij - alpha_i dP_ij)
 * ([FBN] 关键设计 1: the row scalars D, alpha, E and the affine rule for
 * d~P; "FlashBoB: I/O-Efficient Exact Backward-over-Backward for Softmax
 * Attention", paper notes).  These are the same definitions as row_scalars()
 * in oracle/bob.py, which the tests pin against finite differences.
 *
 * Layout: Q, dO, UQ are [Nq][d] and K, V, UK, UV are [Nk][d] row-major float
 * arrays (exact copies of the bf16 or fp32 inputs); L, D, alpha, E are [Nq]
 * double arrays written by the call.
 *
 * Every sum runs over j (or over k for a dot product) in index order, one
 * row at a time, exactly as written above.  Rows are independent: OpenMP
 * hands out groups of RB rows, and the k loops of a group run over the RB
 * rows side by side so that one pass over a key row serves all of them.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define RB 32

/* s[r] = sum_k A[r][k] b[k] for the RB rows of a group (AT is the group's
 * A transposed, AT[k][r], zero past the group's last row); each s[r]
 * accumulates over k in index order. */
static void dots(const double* restrict AT, const float* restrict b, int d,
                 double* restrict s) {
  for (int r = 0; r < RB; ++r) s[r] = 0.0;
  for (int k = 0; k < d; ++k) {
    const double bk = (double)b[k];
    const double* restrict a = AT + (size_t)k * RB;
    for (int r = 0; r < RB; ++r) s[r] += a[r] * bk;
  }
}

static void transpose_rows(const float* X, int i0, int nr, int d, double* XT) {
  for (int k = 0; k < d; ++k)
    for (int r = 0; r < RB; ++r)
      XT[(size_t)k * RB + r] = r < nr ? (double)X[(size_t)(i0 + r) * d + k] : 0.0;
}

int oracle_row_scalars(const float* Q, const float* K, const float* V, const float* dO,
                       const float* UQ, const float* UK, const float* UV, int Nq, int Nk,
                       int d, double tau, int causal, double* L, double* D, double* alpha,
                       double* E) {
  if (Nq <= 0 || Nk <= 0 || d <= 0) return 1;
  const int groups = (Nq + RB - 1) / RB;
  int failed = 0;
#pragma omp parallel
  {
    double* QT = malloc(sizeof(double) * RB * d);
    double* dOT = malloc(sizeof(double) * RB * d);
    double* UQT = malloc(sizeof(double) * RB * d);
    double* O = malloc(sizeof(double) * RB * d);
    double* P = malloc(sizeof(double) * (size_t)RB * Nk); /* S, then P, of the group */
    double* F = malloc(sizeof(double) * (size_t)RB * Nk);
    if (!QT || !dOT || !UQT || !O || !P || !F) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int gi = 0; gi < groups; ++gi) {
        const int i0 = gi * RB, nr = (Nq - i0 < RB) ? Nq - i0 : RB;
        double s[RB], a[RB], b[RB], m[RB], z[RB], Dr[RB], al[RB], Er[RB];
        transpose_rows(Q, i0, nr, d, QT);
        transpose_rows(dO, i0, nr, d, dOT);
        transpose_rows(UQ, i0, nr, d, UQT);
        /* S_ij = tau Q_i.K_j and m_i = max_j S_ij */
        for (int r = 0; r < RB; ++r) m[r] = -INFINITY;
        for (int j = 0; j < Nk; ++j) {
          dots(QT, K + (size_t)j * d, d, s);
          for (int r = 0; r < nr; ++r) {
            const double v = (causal && j > i0 + r) ? -INFINITY : tau * s[r];
            P[(size_t)r * Nk + j] = v;
            if (v > m[r]) m[r] = v;
          }
        }
        /* softmax: P_ij = exp(S_ij - m_i) / z_i, z_i = sum_j exp(S_ij - m_i),
         * and L_i = m_i + log z_i */
        for (int r = 0; r < nr; ++r) {
          double* pr = P + (size_t)r * Nk;
          double zr = 0.0;
          for (int j = 0; j < Nk; ++j) {
            pr[j] = exp(pr[j] - m[r]);
            zr += pr[j];
          }
          for (int j = 0; j < Nk; ++j) pr[j] /= zr;
          z[r] = zr;
          L[i0 + r] = m[r] + log(zr);
        }
        /* F_ij, O_i = sum_j P_ij V_j, alpha_i = sum_j P_ij F_ij */
        memset(O, 0, sizeof(double) * RB * d);
        for (int r = 0; r < RB; ++r) al[r] = 0.0;
        for (int j = 0; j < Nk; ++j) {
          dots(UQT, K + (size_t)j * d, d, a);
          dots(QT, UK + (size_t)j * d, d, b);
          const float* vj = V + (size_t)j * d;
          for (int r = 0; r < nr; ++r) {
            const double p = P[(size_t)r * Nk + j], f = tau * (a[r] + b[r]);
            F[(size_t)r * Nk + j] = f;
            for (int k = 0; k < d; ++k) O[(size_t)r * d + k] += p * (double)vj[k];
            al[r] += p * f;
          }
        }
        for (int r = 0; r < nr; ++r) {
          double acc = 0.0;
          for (int k = 0; k < d; ++k) acc += (double)dO[(size_t)(i0 + r) * d + k] * O[(size_t)r * d + k];
          Dr[r] = acc;
          Er[r] = 0.0;
        }
        /* E_i = sum_j P_ij (F_ij (dP_ij - D_i) + G_ij - alpha_i dP_ij) */
        for (int j = 0; j < Nk; ++j) {
          double dp[RB], g[RB];
          dots(dOT, V + (size_t)j * d, d, dp);
          dots(dOT, UV + (size_t)j * d, d, g);
          for (int r = 0; r < nr; ++r) {
            const double f = F[(size_t)r * Nk + j];
            Er[r] += P[(size_t)r * Nk + j] * (f * (dp[r] - Dr[r]) + g[r] - al[r] * dp[r]);
          }
        }
        for (int r = 0; r < nr; ++r) {
          D[i0 + r] = Dr[r];
          alpha[i0 + r] = al[r];
          E[i0 + r] = Er[r];
        }
        (void)z;
      }
    }
    free(QT);
    free(dOT);
    free(UQT);
    free(O);
    free(P);
    free(F);
  }
  return failed ? 2 : 0;
}
