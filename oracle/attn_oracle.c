/*
 * CPU oracle for exact scaled-dot-product attention, forward and backward, in fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's CPU
 * baseline leg may load this library.  It shares no code with the CUDA path.
 *
 * What it computes is the plain definition the FlashAttention-4 pages reduce to
 * ("Algorithm analysis" page, section 4: O = softmax(QK^T) V computed without the N x N
 * matrix; "FlashAttention-4 explained" page, section 02: every generation computes the
 * same attention, no new mathematics).  Here the N x N scores and probabilities ARE
 * materialised, row by row, in fp64, from the bf16 input values:
 *
 *   S_ij   = scale * sum_k Q_ik K_jk            (S_ij = -inf for j > i when causal)
 *   P_ij   = exp(S_ij - M_i) / sum_j exp(S_ij - M_i),   M_i = max_j S_ij
 *   O_i    = sum_j P_ij V_j
 *   LSE_i  = M_i + ln sum_j exp(S_ij - M_i)      (natural log of the scaled scores)
 *
 * Backward, by the chain rule with upstream gradient dO (the pages' backward stage list,
 * "Hotelren FA4 summary" page section 4.2: S = KQ^T, dP = dO V^T, dV = P^T dO,
 * dS = dsoftmax(dP), dQ += dS K; dK is the fifth product of section 4.1):
 *
 *   dV     = P^T dO
 *   dP     = dO V^T
 *   D_i    = sum_j P_ij dP_ij
 *   dS     = P o (dP - D)
 *   dQ     = scale * dS K
 *   dK     = scale * dS^T Q
 *
 * Grouped heads (GQA/MQA): query head hq reads key/value head hq / (Hq/Hkv); dK and dV
 * of a key/value head are summed over the Hq/Hkv query heads that read it.
 *
 * Layout: Q, dO are [B, Hq, N, d]; K, V are [B, Hkv, N, d]; all bf16 bit patterns
 * (uint16), row-major and contiguous.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_double(uint16_t h) {
  uint32_t bits = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static void load_head(const uint16_t* src, size_t N, size_t d, double* dst) {
  for (size_t i = 0; i < N * d; ++i) dst[i] = bf16_to_double(src[i]);
}

static int check_args(int B, int Hq, int Hkv, int N, int d) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || N < 0 || d <= 0) return -1;
  if (Hq % Hkv != 0) return -1;
  return 0;
}

/* One row i of the probability matrix: fills p[0..N) with P_ij (0 where masked) and
 * returns LSE_i.  qrow and K are fp64 copies. */
static double prob_row(const double* qrow, const double* K, int N, int d, int causal,
                       double scale, int i, double* p) {
  int jend = causal ? i + 1 : N;
  double m = -INFINITY;
  for (int j = 0; j < jend; ++j) {
    double s = 0.0;
    const double* krow = K + (size_t)j * d;
    for (int kk = 0; kk < d; ++kk) s += qrow[kk] * krow[kk];
    s *= scale;
    p[j] = s;
    if (s > m) m = s;
  }
  double sum = 0.0;
  for (int j = 0; j < jend; ++j) {
    p[j] = exp(p[j] - m);
    sum += p[j];
  }
  for (int j = 0; j < jend; ++j) p[j] /= sum;
  for (int j = jend; j < N; ++j) p[j] = 0.0;
  return m + log(sum);
}

/*
 * Forward for a selection of query heads.  sel[s] = b * Hq + hq.  Outputs O[s, N, d] and
 * LSE[s, N] (fp64).  nsel = 0 means nothing to do.  Returns 0, or -1 on bad arguments.
 */
int oracle_attn_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, int B, int Hq,
                    int Hkv, int N, int d, int causal, double scale, int nsel, const int* sel,
                    double* O, double* LSE) {
  if (check_args(B, Hq, Hkv, N, d)) return -1;
  const int g = Hq / Hkv;
  const size_t hd = (size_t)N * d;
  double* Qd = (double*)malloc(hd * sizeof(double) + 1);
  double* Kd = (double*)malloc(hd * sizeof(double) + 1);
  double* Vd = (double*)malloc(hd * sizeof(double) + 1);
  if (!Qd || !Kd || !Vd) {
    free(Qd); free(Kd); free(Vd);
    return -2;
  }
  for (int s = 0; s < nsel; ++s) {
    const int b = sel[s] / Hq, hq = sel[s] % Hq, hkv = hq / g;
    if (b < 0 || b >= B) { free(Qd); free(Kd); free(Vd); return -1; }
    load_head(q + ((size_t)b * Hq + hq) * hd, N, d, Qd);
    load_head(k + ((size_t)b * Hkv + hkv) * hd, N, d, Kd);
    load_head(v + ((size_t)b * Hkv + hkv) * hd, N, d, Vd);
    double* Os = O + (size_t)s * hd;
    double* Ls = LSE + (size_t)s * N;
#pragma omp parallel
    {
      double* p = (double*)malloc(((size_t)N + 1) * sizeof(double));
#pragma omp for schedule(dynamic, 4)
      for (int i = 0; i < N; ++i) {
        Ls[i] = prob_row(Qd + (size_t)i * d, Kd, N, d, causal, scale, i, p);
        double* orow = Os + (size_t)i * d;
        for (int c = 0; c < d; ++c) orow[c] = 0.0;
        for (int j = 0; j < N; ++j) {
          if (p[j] == 0.0) continue;
          const double* vrow = Vd + (size_t)j * d;
          for (int c = 0; c < d; ++c) orow[c] += p[j] * vrow[c];
        }
      }
      free(p);
    }
  }
  free(Qd); free(Kd); free(Vd);
  return 0;
}

/*
 * Backward for a selection of key/value heads.  sel[s] = b * Hkv + hkv.  For each, the g
 * query heads hq = hkv*g .. hkv*g+g-1 are processed.  Outputs dQ[s, g, N, d] and
 * dK[s, N, d], dV[s, N, d] (fp64, dK/dV summed over the group).  P and dS of one query
 * head are held as full N x N fp64 matrices.  Returns 0, -1 on bad arguments, -2 when
 * memory runs out.
 */
int oracle_attn_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                    const uint16_t* dout, int B, int Hq, int Hkv, int N, int d, int causal,
                    double scale, int nsel, const int* sel, double* dQ, double* dK,
                    double* dV) {
  if (check_args(B, Hq, Hkv, N, d)) return -1;
  const int g = Hq / Hkv;
  const size_t hd = (size_t)N * d;
  const size_t nn = (size_t)N * N;
  double* Qd = (double*)malloc(hd * sizeof(double) + 1);
  double* Kd = (double*)malloc(hd * sizeof(double) + 1);
  double* Vd = (double*)malloc(hd * sizeof(double) + 1);
  double* dOd = (double*)malloc(hd * sizeof(double) + 1);
  double* P = (double*)malloc(nn * sizeof(double) + 1);
  double* dS = (double*)malloc(nn * sizeof(double) + 1);
  int rc = 0;
  if (!Qd || !Kd || !Vd || !dOd || !P || !dS) rc = -2;
  for (int s = 0; s < nsel && rc == 0; ++s) {
    const int b = sel[s] / Hkv, hkv = sel[s] % Hkv;
    if (b < 0 || b >= B) { rc = -1; break; }
    load_head(k + ((size_t)b * Hkv + hkv) * hd, N, d, Kd);
    load_head(v + ((size_t)b * Hkv + hkv) * hd, N, d, Vd);
    double* dKs = dK + (size_t)s * hd;
    double* dVs = dV + (size_t)s * hd;
    for (size_t i = 0; i < hd; ++i) { dKs[i] = 0.0; dVs[i] = 0.0; }
    for (int r = 0; r < g; ++r) {
      const int hq = hkv * g + r;
      load_head(q + ((size_t)b * Hq + hq) * hd, N, d, Qd);
      load_head(dout + ((size_t)b * Hq + hq) * hd, N, d, dOd);
      double* dQs = dQ + ((size_t)s * g + r) * hd;
      /* Rows: P_i, dP_i = dO_i V^T, D_i, dS_i, dQ_i = scale * dS_i K. */
#pragma omp parallel
      {
        double* dp = (double*)malloc(((size_t)N + 1) * sizeof(double));
#pragma omp for schedule(dynamic, 4)
        for (int i = 0; i < N; ++i) {
          double* prow = P + (size_t)i * N;
          double* dsrow = dS + (size_t)i * N;
          prob_row(Qd + (size_t)i * d, Kd, N, d, causal, scale, i, prow);
          const double* dorow = dOd + (size_t)i * d;
          double D = 0.0;
          for (int j = 0; j < N; ++j) {
            const double* vrow = Vd + (size_t)j * d;
            double acc = 0.0;
            for (int c = 0; c < d; ++c) acc += dorow[c] * vrow[c];
            dp[j] = acc;
            D += prow[j] * acc;
          }
          for (int j = 0; j < N; ++j) dsrow[j] = prow[j] * (dp[j] - D);
          double* dqrow = dQs + (size_t)i * d;
          for (int c = 0; c < d; ++c) dqrow[c] = 0.0;
          for (int j = 0; j < N; ++j) {
            if (dsrow[j] == 0.0) continue;
            const double* krow = Kd + (size_t)j * d;
            for (int c = 0; c < d; ++c) dqrow[c] += dsrow[j] * krow[c];
          }
          for (int c = 0; c < d; ++c) dqrow[c] *= scale;
        }
        free(dp);
      }
      /* Columns: dV_j += sum_i P_ij dO_i ; dK_j += scale * sum_i dS_ij Q_i. */
#pragma omp parallel for schedule(dynamic, 4)
      for (int j = 0; j < N; ++j) {
        double* dvrow = dVs + (size_t)j * d;
        double* dkrow = dKs + (size_t)j * d;
        for (int i = 0; i < N; ++i) {
          const double pij = P[(size_t)i * N + j];
          const double sij = dS[(size_t)i * N + j];
          if (pij != 0.0) {
            const double* dorow = dOd + (size_t)i * d;
            for (int c = 0; c < d; ++c) dvrow[c] += pij * dorow[c];
          }
          if (sij != 0.0) {
            const double* qrow = Qd + (size_t)i * d;
            for (int c = 0; c < d; ++c) dkrow[c] += scale * sij * qrow[c];
          }
        }
      }
    }
  }
  free(Qd); free(Kd); free(Vd); free(dOd); free(P); free(dS);
  return rc;
}

/*
 * Forward with a key/value sequence longer than the query sequence (queries appended
 * after a cache of keys): q [B,Hq,Nq,d], k/v [B,Hkv,Nk,d].  Query i stands at position
 * i + (Nk - Nq) of the key sequence, so with causal it sees keys j <= i + Nk - Nq
 * (the mask aligned at the bottom-right corner; Nq = Nk is the square case above).
 * Causal needs Nq <= Nk (every query sees at least one key).  sel[s] = b * Hq + hq;
 * outputs O[s, Nq, d] and LSE[s, Nq].  Returns 0, -1 on bad arguments, -2 without memory.
 */
int oracle_attn_fwd_kv(const uint16_t* q, const uint16_t* k, const uint16_t* v, int B, int Hq, int Hkv, int Nq,
                       int Nk, int d, int causal, double scale, int nsel, const int* sel, double* O, double* LSE) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Nq < 0 || Nk < 0 || d <= 0 || Hq % Hkv != 0) return -1;
  if (causal && Nq > Nk) return -1;
  const int g = Hq / Hkv;
  const int off = Nk - Nq;
  const size_t qd = (size_t)Nq * d, kd = (size_t)Nk * d;
  double* Qd = (double*)malloc(qd * sizeof(double) + 1);
  double* Kd = (double*)malloc(kd * sizeof(double) + 1);
  double* Vd = (double*)malloc(kd * sizeof(double) + 1);
  if (!Qd || !Kd || !Vd) {
    free(Qd); free(Kd); free(Vd);
    return -2;
  }
  int rc = 0;
  for (int s = 0; s < nsel && rc == 0; ++s) {
    const int b = sel[s] / Hq, hq = sel[s] % Hq, hkv = hq / g;
    if (b < 0 || b >= B) { rc = -1; break; }
    load_head(q + ((size_t)b * Hq + hq) * qd, Nq, d, Qd);
    load_head(k + ((size_t)b * Hkv + hkv) * kd, Nk, d, Kd);
    load_head(v + ((size_t)b * Hkv + hkv) * kd, Nk, d, Vd);
    double* Os = O + (size_t)s * qd;
    double* Ls = LSE + (size_t)s * Nq;
#pragma omp parallel
    {
      double* p = (double*)malloc(((size_t)Nk + 1) * sizeof(double));
#pragma omp for schedule(dynamic, 4)
      for (int i = 0; i < Nq; ++i) {
        const int jend = causal ? i + off + 1 : Nk;   /* keys [0, jend) are visible */
        const double* qrow = Qd + (size_t)i * d;
        double m = -INFINITY;
        for (int j = 0; j < jend; ++j) {
          double sc = 0.0;
          const double* krow = Kd + (size_t)j * d;
          for (int kk = 0; kk < d; ++kk) sc += qrow[kk] * krow[kk];
          p[j] = sc * scale;
          if (p[j] > m) m = p[j];
        }
        double sum = 0.0;
        for (int j = 0; j < jend; ++j) {
          p[j] = exp(p[j] - m);
          sum += p[j];
        }
        double* orow = Os + (size_t)i * d;
        for (int c = 0; c < d; ++c) orow[c] = 0.0;
        for (int j = 0; j < jend; ++j) {
          const double w = p[j] / sum;
          const double* vrow = Vd + (size_t)j * d;
          for (int c = 0; c < d; ++c) orow[c] += w * vrow[c];
        }
        Ls[i] = m + log(sum);
      }
      free(p);
    }
  }
  free(Qd); free(Kd); free(Vd);
  return rc;
}
