/*
 * ssd_oracle.c -- plain double-precision CPU oracle for the Mamba2 SSD ops.
 *
 * TEST INFRASTRUCTURE ONLY (see ssd_oracle.h): used by the tests, the package smoke
 * check and the benchmark's CPU-baseline leg; never by the product path.
 *
 * Built with -O2 -ffp-contract=off (no fused multiply-add contraction, no fast-math)
 * so that every operation rounds once in double, as written.  OpenMP only spreads
 * independent (sequence, head) or (row, head) units over host cores; each unit is a
 * plain loop in the order written.
 *
 * Mutation points (ORACLE_MUTANT), from the vllm.cpp page "W2 finish
 * (KERNEL-SSM-MAMBA)", section "Evidence", mutation table:
 *   M1 drop the inter-chunk state term      M2 ignore initial_states
 *   M3 read states[c] for states[c-1]       M4 drop the D skip connection
 *   M5 ignore state_indices                 M6 NULL row as slot 0
 *   M7 whole-row variance, not per-group    M8 sigmoid instead of silu
 *   M9 drop the decode A < 0 check
 */
#include "ssd_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* softplus(v) = log(1 + e^v); above 20 the difference from v is below double's
 * resolution relative to v (e^-20 ~ 2e-9 absolute, and the GPU computes in fp32). */
static double softplus(double v) { return v > 20.0 ? v : log1p(exp(v)); }

static double dt_of(double raw, const double* dt_bias, int h, int dt_softplus) {
  double v = raw + (dt_bias ? dt_bias[h] : 0.0);
  return dt_softplus ? softplus(v) : v;
}

static int check_meta(const int32_t* cu, int nseq, int T) {
  if (nseq < 1 || !cu || cu[0] != 0 || cu[nseq] != T) return 0;
  for (int s = 0; s < nseq; ++s)
    if (cu[s + 1] < cu[s]) return 0;
  return 1;
}

/* ---------------------------------------------------------------------------- */
/* Sequential recurrence: the definition, token by token.                        */
/* ---------------------------------------------------------------------------- */
int oracle_scan_seq(const double* x, const double* dt_raw, const double* dt_bias,
                    int dt_softplus, const double* A, const double* B, const double* C,
                    const double* D, const double* init, const uint8_t* has_init,
                    const int32_t* cu, int nseq, int T, int H, int P, int G, int N,
                    double* y, double* final_states, double* y_abs, double* final_abs) {
  if (!x || !dt_raw || !A || !B || !C || !y || H < 1 || G < 1 || H % G || P < 1 || N < 1)
    return ORACLE_BAD_ARG;
  if (!check_meta(cu, nseq, T)) return ORACLE_BAD_ARG;
  const int hpg = H / G;
  const size_t PN = (size_t)P * N;

#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int s = 0; s < nseq; ++s) {
    for (int h = 0; h < H; ++h) {
      const int g = h / hpg;
      double* st = (double*)malloc(PN * sizeof(double));
      double* sa = (double*)malloc(PN * sizeof(double));
      const int use_init = init && (!has_init || has_init[s]) && ORACLE_MUTANT != 2;
      for (size_t e = 0; e < PN; ++e) {
        double v = use_init ? init[((size_t)s * H + h) * PN + e] : 0.0;
        st[e] = v;
        sa[e] = fabs(v);
      }
      const double Dh = D ? D[h] : 0.0;
      for (int t = cu[s]; t < cu[s + 1]; ++t) {
        const double dt = dt_of(dt_raw[(size_t)t * H + h], dt_bias, h, dt_softplus);
        const double a = exp(dt * A[h]);
        const double* Bt = B + ((size_t)t * G + g) * N;
        const double* Ct = C + ((size_t)t * G + g) * N;
        for (int p = 0; p < P; ++p) {
          const double xv = x[((size_t)t * H + h) * P + p];
          double acc = 0.0, acc_abs = 0.0;
          for (int n = 0; n < N; ++n) {
            double* hp = st + (size_t)p * N + n;
            *hp = a * (*hp) + dt * Bt[n] * xv;
            acc += Ct[n] * (*hp);
            double* ha = sa + (size_t)p * N + n;
            *ha = a * (*ha) + fabs(dt * Bt[n] * xv);
            acc_abs += fabs(Ct[n]) * (*ha);
          }
          double dterm = (ORACLE_MUTANT == 4) ? 0.0 : Dh * xv;
          y[((size_t)t * H + h) * P + p] = acc + dterm;
          if (y_abs) y_abs[((size_t)t * H + h) * P + p] = acc_abs + fabs(dterm);
        }
      }
      if (final_states)
        memcpy(final_states + ((size_t)s * H + h) * PN, st, PN * sizeof(double));
      if (final_abs) memcpy(final_abs + ((size_t)s * H + h) * PN, sa, PN * sizeof(double));
      free(st);
      free(sa);
    }
  }
  return ORACLE_OK;
}

/* ---------------------------------------------------------------------------- */
/* Chunked restatement.  Per sequence and head, chunks of Q tokens starting at the  */
/* sequence start (the last one partial).  Within chunk c, with a_t = dt_t*A and   */
/* cs_i = sum_{r<=i in chunk} a_r:                                                 */
/*   CB[i,j]   = sum_n C_i[n] B_j[n]                                               */
/*   Ydiag[i]  = sum_{j<=i} CB[i,j] * exp(cs_i - cs_j) * dt_j * x_j                 */
/*   Yoff[i]   = exp(cs_i) * sum_n C_i[n] * h_{c-1}[:,n]                           */
/*   y_i       = Ydiag + Yoff + D x_i                                              */
/*   S_c[p,n]  = sum_j exp(cs_last - cs_j) * dt_j * x_j[p] * B_j[n]                 */
/*   h_c       = exp(cs_last) * h_{c-1} + S_c     (h_{-1} = initial state or 0)     */
/* ---------------------------------------------------------------------------- */
int oracle_scan_chunked(const double* x, const double* dt_raw, const double* dt_bias,
                        int dt_softplus, const double* A, const double* B, const double* C,
                        const double* D, const double* init, const uint8_t* has_init,
                        const int32_t* cu, int nseq, int T, int H, int P, int G, int N,
                        int Q, double* y, double* final_states) {
  if (!x || !dt_raw || !A || !B || !C || !y || H < 1 || G < 1 || H % G || P < 1 || N < 1 ||
      Q < 1)
    return ORACLE_BAD_ARG;
  if (!check_meta(cu, nseq, T)) return ORACLE_BAD_ARG;
  const int hpg = H / G;
  const size_t PN = (size_t)P * N;

#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int s = 0; s < nseq; ++s) {
    for (int h = 0; h < H; ++h) {
      const int g = h / hpg;
      double* hprev = (double*)malloc(PN * sizeof(double));
      double* hnew = (double*)malloc(PN * sizeof(double));
      double* cs = (double*)malloc((size_t)Q * sizeof(double));
      double* dtv = (double*)malloc((size_t)Q * sizeof(double));
      const int use_init = init && (!has_init || has_init[s]) && ORACLE_MUTANT != 2;
      for (size_t e = 0; e < PN; ++e)
        hprev[e] = use_init ? init[((size_t)s * H + h) * PN + e] : 0.0;
      const double Dh = D ? D[h] : 0.0;
      for (int c0 = cu[s]; c0 < cu[s + 1]; c0 += Q) {
        const int len = (cu[s + 1] - c0 < Q) ? cu[s + 1] - c0 : Q;
        /* dt and the within-chunk cumulative sum of dt*A */
        double run = 0.0;
        for (int i = 0; i < len; ++i) {
          dtv[i] = dt_of(dt_raw[(size_t)(c0 + i) * H + h], dt_bias, h, dt_softplus);
          run += dtv[i] * A[h];
          cs[i] = run;
        }
        const double cs_last = cs[len - 1];
        /* chunk state S_c, then h_c = exp(cs_last) h_{c-1} + S_c */
        for (int p = 0; p < P; ++p)
          for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int j = 0; j < len; ++j) {
              const int t = c0 + j;
              acc += exp(cs_last - cs[j]) * dtv[j] * x[((size_t)t * H + h) * P + p] *
                     B[((size_t)t * G + g) * N + n];
            }
            hnew[(size_t)p * N + n] = exp(cs_last) * hprev[(size_t)p * N + n] + acc;
          }
        /* outputs: the state entering the chunk is h_{c-1} (M3 reads h_c instead) */
        const double* hin = (ORACLE_MUTANT == 3) ? hnew : hprev;
        for (int i = 0; i < len; ++i) {
          const int ti = c0 + i;
          const double* Ci = C + ((size_t)ti * G + g) * N;
          for (int p = 0; p < P; ++p) {
            double ydiag = 0.0;
            for (int j = 0; j <= i; ++j) {
              const int tj = c0 + j;
              const double* Bj = B + ((size_t)tj * G + g) * N;
              double cb = 0.0;
              for (int n = 0; n < N; ++n) cb += Ci[n] * Bj[n];
              ydiag += cb * exp(cs[i] - cs[j]) * dtv[j] * x[((size_t)tj * H + h) * P + p];
            }
            double yoff = 0.0;
            for (int n = 0; n < N; ++n) yoff += Ci[n] * hin[(size_t)p * N + n];
            yoff *= exp(cs[i]);
            if (ORACLE_MUTANT == 1) yoff *= 0.0;
            const double xv = x[((size_t)ti * H + h) * P + p];
            const double dterm = (ORACLE_MUTANT == 4) ? 0.0 : Dh * xv;
            y[((size_t)ti * H + h) * P + p] = ydiag + yoff + dterm;
          }
        }
        double* tmp = hprev;
        hprev = hnew;
        hnew = tmp;
      }
      if (final_states)
        memcpy(final_states + ((size_t)s * H + h) * PN, hprev, PN * sizeof(double));
      free(hprev);
      free(hnew);
      free(cs);
      free(dtv);
    }
  }
  return ORACLE_OK;
}

/* ---------------------------------------------------------------------------- */
/* Decode: one recurrence step on a pooled state slot per batch row.              */
/* ---------------------------------------------------------------------------- */
int oracle_state_update(double* pool, int num_slots, const int32_t* idx, int batch,
                        const double* x, const double* dt_raw, const double* dt_bias,
                        int dt_softplus, const double* A, const double* B, const double* C,
                        const double* D, int H, int P, int G, int N, double* y,
                        int32_t* status) {
  if (!pool || !idx || !x || !dt_raw || !A || !B || !C || !y || H < 1 || G < 1 || H % G ||
      P < 1 || N < 1 || num_slots < 1 || batch < 0)
    return ORACLE_BAD_ARG;
  const int hpg = H / G;
  const size_t PN = (size_t)P * N;
  int32_t st = 0;

  /* index and sign checks first (they decide what may be written) */
  for (int b = 0; b < batch; ++b) {
    int s = idx[b];
    if (ORACLE_MUTANT == 5) s = b;
    if (s < -1 || s >= num_slots) st |= ORACLE_ST_INDEX_OOR;
  }
  for (int h = 0; h < H; ++h)
    if (!(A[h] < 0.0) && ORACLE_MUTANT != 9) st |= ORACLE_ST_A_NOT_NEG;

#pragma omp parallel for collapse(2) schedule(static)
  for (int b = 0; b < batch; ++b) {
    for (int h = 0; h < H; ++h) {
      int s = idx[b];
      if (ORACLE_MUTANT == 5) s = b;
      if (ORACLE_MUTANT == 6 && s == -1) s = 0;
      double* yb = y + ((size_t)b * H + h) * P;
      const int a_ok = (A[h] < 0.0) || ORACLE_MUTANT == 9;
      if (s < 0 || s >= num_slots || !a_ok) {
        for (int p = 0; p < P; ++p) yb[p] = 0.0;
        continue;
      }
      const int g = h / hpg;
      const double dt = dt_of(dt_raw[(size_t)b * H + h], dt_bias, h, dt_softplus);
      const double a = exp(dt * A[h]);
      const double* Bb = B + ((size_t)b * G + g) * N;
      const double* Cb = C + ((size_t)b * G + g) * N;
      double* S = pool + ((size_t)s * H + h) * PN;
      const double Dh = D ? D[h] : 0.0;
      for (int p = 0; p < P; ++p) {
        const double xv = x[((size_t)b * H + h) * P + p];
        double acc = 0.0;
        for (int n = 0; n < N; ++n) {
          double* e = S + (size_t)p * N + n;
          *e = a * (*e) + dt * Bb[n] * xv;
          acc += Cb[n] * (*e);
        }
        yb[p] = acc + ((ORACLE_MUTANT == 4) ? 0.0 : Dh * xv);
      }
    }
  }
  if (status) *status = st;
  return ORACLE_OK;
}

/* ---------------------------------------------------------------------------- */
/* Gated RMSNorm, gate first: out = norm(x * silu(z)) * w, variance per group.     */
/* ---------------------------------------------------------------------------- */
static double gate(double z) {
  double sig = 1.0 / (1.0 + exp(-z));
  return (ORACLE_MUTANT == 8) ? sig : z * sig;
}

int oracle_gated_rmsnorm(const double* x, const double* z, const double* w, double* out,
                         int64_t rows, int d, int group_size, double eps) {
  if (!x || !w || !out || rows < 0 || d < 1 || group_size < 1 || d % group_size) return ORACLE_BAD_ARG;
  /* M7 computes one variance over the whole row (every variable still read) */
  const int gs = (ORACLE_MUTANT == 7) ? d : group_size;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const double* xr = x + (size_t)r * d;
    const double* zr = z ? z + (size_t)r * d : NULL;
    double* orow = out + (size_t)r * d;
    for (int g0 = 0; g0 < d; g0 += gs) {
      double ss = 0.0;
      for (int k = g0; k < g0 + gs; ++k) {
        double g = zr ? xr[k] * gate(zr[k]) : xr[k];
        ss += g * g;
      }
      const double rinv = 1.0 / sqrt(ss / gs + eps);
      for (int k = g0; k < g0 + gs; ++k) {
        double g = zr ? xr[k] * gate(zr[k]) : xr[k];
        orow[k] = g * rinv * w[k];
      }
    }
  }
  return ORACLE_OK;
}
