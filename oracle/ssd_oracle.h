/*
 * ssd_oracle.h -- plain double-precision CPU oracle for the three Mamba2 SSD ops.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path (the CUDA library, its
 * Python binding) may include, link or call this code; only the test suite, the
 * package's smoke check and the benchmark's CPU-baseline leg use it.  It shares no
 * code, header, table or helper with the CUDA path.
 *
 * What it computes (the op names are those of the vllm.cpp page "W2 finish
 * (KERNEL-SSM-MAMBA)", PR #566 / #675: vt::Mamba2ChunkScan, vt::Mamba2StateUpdate,
 * vt::RmsNormGatedGroup):
 *
 *   Mamba2 SSD recurrence (Dao & Gu, "Transformers are SSMs", 2024, the SSD layer),
 *   per sequence, head h (group g = h / (H/G)), channel p, state index n:
 *     dt_t     = softplus(dt_raw[t,h] + dt_bias[h])      (or the plain sum if softplus is off)
 *     h_t[p,n] = exp(dt_t*A[h]) * h_{t-1}[p,n] + dt_t * B[t,g,n] * x[t,h,p]
 *     y[t,h,p] = sum_n C[t,g,n] * h_t[p,n] + D[h] * x[t,h,p]
 *   with h_{-1} = initial_states[s] when present, else 0; final_states[s] = h at the
 *   sequence's last token.
 *
 * Everything is computed in double from the caller's values.  No blocking, fusion or
 * reordering beyond what each function's comment states.
 *
 * Compile-time ORACLE_MUTANT=k (1..9) plants the pages' mutation k (page above,
 * section "Evidence", mutation table) into this oracle so that the test suite can
 * show its pins catch it.  The pristine build has ORACLE_MUTANT undefined.
 */
#ifndef SSD_ORACLE_H
#define SSD_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* return codes */
#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1

/* status bits reported by the decode oracle (same meaning as the library's, but
 * defined independently here) */
#define ORACLE_ST_A_NOT_NEG 1
#define ORACLE_ST_INDEX_OOR 2

/* Sequential recurrence -- the definition.  Layouts (row-major, dense):
 *   x [T,H,P]; dt_raw [T,H]; dt_bias [H] (NULL = 0); A [H]; B, C [T,G,N]; D [H] (NULL = 0)
 *   init [nseq,H,P,N] (NULL = zero); has_init [nseq] (NULL = all 1 when init != NULL)
 *   cu_seqlens [nseq+1], non-decreasing, cu[0] = 0, cu[nseq] = T
 *   y [T,H,P] out; final_states [nseq,H,P,N] out (NULL = not written)
 * When y_abs / final_abs are non-NULL the same recurrence is also evaluated on
 * absolute values of every term (the summation-error scale sum|terms|). */
int oracle_scan_seq(const double* x, const double* dt_raw, const double* dt_bias,
                    int dt_softplus, const double* A, const double* B, const double* C,
                    const double* D, const double* init, const uint8_t* has_init,
                    const int32_t* cu_seqlens, int nseq, int T, int H, int P, int G, int N,
                    double* y, double* final_states, double* y_abs, double* final_abs);

/* The chunked restatement (segsum decay, C.B^T, chunk states, state passing, output
 * contractions), chunk length Q, chunks restarting at each sequence start.  Exact
 * arithmetic gives the sequential result for any Q. */
int oracle_scan_chunked(const double* x, const double* dt_raw, const double* dt_bias,
                        int dt_softplus, const double* A, const double* B, const double* C,
                        const double* D, const double* init, const uint8_t* has_init,
                        const int32_t* cu_seqlens, int nseq, int T, int H, int P, int G,
                        int N, int Q, double* y, double* final_states);

/* One decode token per batch row b: pool slot s = state_indices[b].
 *   pool [num_slots,H,P,N] (updated in place); x [batch,H,P]; dt_raw [batch,H];
 *   B, C [batch,G,N]; y [batch,H,P] out.
 * s == -1: the row touches no slot and y[b] = 0.  s outside [-1, num_slots): status
 * ORACLE_ST_INDEX_OOR, no slot touched, y[b] = 0.  A[h] not < 0 (including +0, -0
 * and NaN): status ORACLE_ST_A_NOT_NEG, that (b,h) leaves the slot untouched and
 * y[b,h,:] = 0.  Returns the OR of the status bits in *status (may be NULL). */
int oracle_state_update(double* pool, int num_slots, const int32_t* state_indices, int batch,
                        const double* x, const double* dt_raw, const double* dt_bias,
                        int dt_softplus, const double* A, const double* B, const double* C,
                        const double* D, int H, int P, int G, int N, double* y,
                        int32_t* status);

/* Gated RMSNorm with per-group variance:
 *   g = x * silu(z) (z NULL = no gate), silu(z) = z / (1 + exp(-z));
 *   per row and each group of group_size contiguous channels:
 *   out = g / sqrt(mean(g^2) + eps) * weight.
 *   x, z, out [rows, d]; weight [d]. */
int oracle_gated_rmsnorm(const double* x, const double* z, const double* weight, double* out,
                         int64_t rows, int d, int group_size, double eps);

#ifdef __cplusplus
}
#endif
#endif
