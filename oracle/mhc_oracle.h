/*
 * fp64 CPU oracle of the mHC forward pass — TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this library.  It is a plain, single-threaded, obviously correct
 * restatement of the equations on the page "mHC 算法分析 & cutile 高效实现"
 * (§2.1–§2.5), with no blocking, fusion or reordering beyond what the
 * equations state.  It shares no code with the CUDA library.
 *
 * Conventions (all arrays row-major, caller-owned host memory):
 *   B tokens, expansion n (1..8), hidden size C, K = n*C, N = n*n + 2*n.
 *   bf16 inputs are passed as their 16-bit patterns and widened exactly.
 *   X     [B][K]  bf16   stream i of token b is X[b][i*C .. i*C+C-1]
 *   phi   [K][N]  bf16   the projection φ in its mathematical orientation
 *   F_out [B][C]  bf16
 *   bias  [N]     double column order: pre [0,n), post [n,2n), res [2n, N)
 *   Y     [B][N]  double raw coefficients  Ỹ = X·φ
 *   r     [B]     double RMS scale
 *   Ht    [B][N]  double scaled coefficients H̃ = α·Ỹ/r + b
 *   H_pre [B][n], H_post [B][n], H_res [B][n][n] (row i = output stream)
 *   F_pre [B][C], X_next [B][K]  double (not rounded)
 */
#ifndef MHC_ORACLE_H
#define MHC_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

double oracle_bf16_to_f64(uint16_t bits);

void oracle_gemm_rms(const uint16_t *X, const uint16_t *phi, int64_t B, int n, int64_t C,
                     double *Y, double *r);

void oracle_scale_bias(const double *Y, const double *r, double a_pre, double a_post,
                       double a_res, const double *bias, int64_t B, int n, double *Ht);

void oracle_sinkhorn(const double *Ht_res, int n, int iters, double *H_res);

void oracle_constraints(const double *Ht, int iters, int64_t B, int n, double *H_pre,
                        double *H_post, double *H_res);

void oracle_coeffs(const double *Y, const double *r, double a_pre, double a_post, double a_res,
                   const double *bias, int iters, int64_t B, int n, double *H_pre,
                   double *H_post, double *H_res);

void oracle_pre_apply(const uint16_t *X, const double *H_pre, int64_t B, int n, int64_t C,
                      double *F_pre);

void oracle_post_res_apply(const uint16_t *X, const uint16_t *F_out, const double *H_res,
                           const double *H_post, int64_t B, int n, int64_t C, double *X_next);

void oracle_forward(const uint16_t *X, const uint16_t *phi, const uint16_t *F_out, int64_t B,
                    int n, int64_t C, double a_pre, double a_post, double a_res,
                    const double *bias, int iters, double *Y, double *r, double *H_pre,
                    double *H_post, double *H_res, double *F_pre, double *X_next);

/* "Towards Free Normalization" §2: C = rmsnorm(A) @ B with eps inside the
 * square root.  A [M][K] bf16 bits, Bm [K][N] bf16 bits, C [M][N] double. */
void oracle_rmsnorm_gemm(const uint16_t *A, const uint16_t *Bm, int64_t M, int64_t K, int64_t N,
                         double eps, double *Cout);

/* fp32 weight / fp32 F_out variants (the page's §5 benchmark precision):
 * φ [K][N] and F_out [B][C] as doubles. */
void oracle_gemm_rms_f64phi(const uint16_t *X, const double *phi, int64_t B, int n, int64_t C,
                            double *Y, double *r);
void oracle_post_res_apply_f64F(const uint16_t *X, const double *F_out, const double *H_res,
                                const double *H_post, int64_t B, int n, int64_t C,
                                double *X_next);
void oracle_forward_f64w(const uint16_t *X, const double *phi, const double *F_out, int64_t B,
                         int n, int64_t C, double a_pre, double a_post, double a_res,
                         const double *bias, int iters, double *Y, double *r, double *H_pre,
                         double *H_post, double *H_res, double *F_pre, double *X_next);

/* fp8 e4m3 (the page's §4 benchmark precision): decode, and the forward with
 * X [B][K], φ [K][N], F_out [B][C] as e4m3 codes. */
double oracle_e4m3_to_f64(uint8_t b);
void oracle_forward_e4m3(const uint8_t *X, const uint8_t *phi, const uint8_t *F_out, int64_t B,
                         int n, int64_t C, double a_pre, double a_post, double a_res,
                         const double *bias, int iters, double *Y, double *r, double *H_pre,
                         double *H_post, double *H_res, double *F_pre, double *X_next);

#ifdef __cplusplus
}
#endif

#endif /* MHC_ORACLE_H */
