/*
 * fp64 CPU oracle of the mHC forward pass — TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this file's library; the product path never does.  Every function is
 * a direct, single-threaded restatement of one equation group on the page
 * "mHC 算法分析 & cutile 高效实现" (mHC algorithm analysis and an efficient
 * cuTile implementation), §2.1–§2.5.  Sums run in index order in double
 * precision.  See mhc_oracle.h for shapes and layouts.
 *
 * Readings taken where the page is silent or garbled:
 *   - r has no epsilon (§2.2 and the r computation of §4.1 add none);
 *   - sigmoid(x) = 1 / (1 + exp(-x)) (§2.4; the helper's body is not shown);
 *   - Sinkhorn starts from exp(H̃_res) and each iteration normalises the rows,
 *     then the columns (§2.4, and the loop order of §4.3 / §5.3); iters = 0
 *     returns exp(H̃_res) unnormalised;
 *   - H_res row i mixes into output stream i: X_next[i] = Σ_j H_res[i][j]·X[j]
 *     (§3.4 and §5.4), and "H_post^T · F_out" is the per-token outer product
 *     X_post[i][c] = H_post[i]·F_out[c] (§3.4 loop, §5.4).
 *
 * oracle_rmsnorm_gemm restates a second page, "Towards Free Normalization:
 * Fusing Normalization into GEMM and Attention Kernels" (PyTorch blog), §2:
 * C = rmsnorm(A) @ B with rmsnorm(A) = A · rstd(A) row by row and
 * rstd = 1 / sqrt(mean of the row's squares + eps).  It is written as that
 * definition (normalise first, then multiply), not in the page's lazy order.
 */
#include "mhc_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* bf16 is the upper half of an IEEE binary32: widening is exact. */
double oracle_bf16_to_f64(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * §2.1: one GEMM gives every raw coefficient, Ỹ = X_t · φ_t, with
 *       φ_t ∈ R^{nC × (n²+2n)}.
 * §2.2: r = sqrt( Σ X_t² / (nC) ), one scalar per token.
 */
void oracle_gemm_rms(const uint16_t *X, const uint16_t *phi, int64_t B, int n, int64_t C,
                     double *Y, double *r)
{
    const int64_t K = (int64_t)n * C;
    const int N = n * n + 2 * n;
    for (int64_t b = 0; b < B; ++b) {
        const uint16_t *x = X + b * K;
        for (int k = 0; k < N; ++k) {
            double acc = 0.0;
            for (int64_t q = 0; q < K; ++q)
                acc += oracle_bf16_to_f64(x[q]) * oracle_bf16_to_f64(phi[q * N + k]);
            Y[b * N + k] = acc;
        }
        double ss = 0.0;
        for (int64_t q = 0; q < K; ++q) {
            double v = oracle_bf16_to_f64(x[q]);
            ss += v * v;
        }
        r[b] = sqrt(ss / (double)K);
    }
}

/*
 * §2.3: H̃_pre = α_pre·Ỹ_pre / r + b_pre, and likewise for post and res.
 * Columns [0,n) are pre, [n,2n) post, [2n, n²+2n) res (res row-major n×n).
 */
void oracle_scale_bias(const double *Y, const double *r, double a_pre, double a_post,
                       double a_res, const double *bias, int64_t B, int n, double *Ht)
{
    const int N = n * n + 2 * n;
    for (int64_t b = 0; b < B; ++b) {
        for (int k = 0; k < N; ++k) {
            double alpha = k < n ? a_pre : (k < 2 * n ? a_post : a_res);
            Ht[b * N + k] = alpha * Y[b * N + k] / r[b] + bias[k];
        }
    }
}

/*
 * §2.4, Sinkhorn–Knopp: start from exp(H̃_res), then repeat `iters` times:
 * divide every row by its sum, then divide every column by its sum.
 * Ht_res and H_res are one token's n×n block, row-major.
 */
void oracle_sinkhorn(const double *Ht_res, int n, int iters, double *H_res)
{
    for (int i = 0; i < n * n; ++i)
        H_res[i] = exp(Ht_res[i]);
    for (int t = 0; t < iters; ++t) {
        for (int i = 0; i < n; ++i) {
            double s = 0.0;
            for (int j = 0; j < n; ++j)
                s += H_res[i * n + j];
            for (int j = 0; j < n; ++j)
                H_res[i * n + j] /= s;
        }
        for (int j = 0; j < n; ++j) {
            double s = 0.0;
            for (int i = 0; i < n; ++i)
                s += H_res[i * n + j];
            for (int i = 0; i < n; ++i)
                H_res[i * n + j] /= s;
        }
    }
}

/*
 * §2.4 constraints: H_pre = sigmoid(H̃_pre), H_post = 2·sigmoid(H̃_post),
 * H_res = Sinkhorn–Knopp(H̃_res).
 */
void oracle_constraints(const double *Ht, int iters, int64_t B, int n, double *H_pre,
                        double *H_post, double *H_res)
{
    const int N = n * n + 2 * n;
    for (int64_t b = 0; b < B; ++b) {
        const double *h = Ht + b * N;
        for (int i = 0; i < n; ++i) {
            H_pre[b * n + i] = 1.0 / (1.0 + exp(-h[i]));
            H_post[b * n + i] = 2.0 / (1.0 + exp(-h[n + i]));
        }
        oracle_sinkhorn(h + 2 * n, n, iters, H_res + b * n * n);
    }
}

/* §2.3 followed by §2.4, token by token. */
void oracle_coeffs(const double *Y, const double *r, double a_pre, double a_post, double a_res,
                   const double *bias, int iters, int64_t B, int n, double *H_pre,
                   double *H_post, double *H_res)
{
    const int N = n * n + 2 * n;
    double Ht[80];
    for (int64_t b = 0; b < B; ++b) {
        oracle_scale_bias(Y + b * N, r + b, a_pre, a_post, a_res, bias, 1, n, Ht);
        oracle_constraints(Ht, iters, 1, n, H_pre + b * n, H_post + b * n, H_res + b * n * n);
    }
}

/* §2.5 (1), Pre (n → 1): F_pre = Σ_i H_pre[i] · X_t[i]. */
void oracle_pre_apply(const uint16_t *X, const double *H_pre, int64_t B, int n, int64_t C,
                      double *F_pre)
{
    const int64_t K = (int64_t)n * C;
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t c = 0; c < C; ++c) {
            double acc = 0.0;
            for (int i = 0; i < n; ++i)
                acc += H_pre[b * n + i] * oracle_bf16_to_f64(X[b * K + (int64_t)i * C + c]);
            F_pre[b * C + c] = acc;
        }
    }
}

/*
 * §2.5 (3), Post & Res: X_res = H_res · X_t, X_post = H_post^T · F_out,
 * X_{t+1} = X_res + X_post, i.e. for every token, stream i and channel c:
 *   X_next[i][c] = Σ_j H_res[i][j]·X[j][c] + H_post[i]·F_out[c].
 */
void oracle_post_res_apply(const uint16_t *X, const uint16_t *F_out, const double *H_res,
                           const double *H_post, int64_t B, int n, int64_t C, double *X_next)
{
    const int64_t K = (int64_t)n * C;
    for (int64_t b = 0; b < B; ++b) {
        const double *h = H_res + b * n * n;
        for (int i = 0; i < n; ++i) {
            for (int64_t c = 0; c < C; ++c) {
                double x_res = 0.0;
                for (int j = 0; j < n; ++j)
                    x_res += h[i * n + j] * oracle_bf16_to_f64(X[b * K + (int64_t)j * C + c]);
                double x_post = H_post[b * n + i] * oracle_bf16_to_f64(F_out[b * C + c]);
                X_next[b * K + (int64_t)i * C + c] = x_res + x_post;
            }
        }
    }
}

/*
 * The whole forward of §2, with F_out taken as an input: the layer function
 * F between F_pre and F_out (§2.5 (2)) lies outside mHC.
 */
void oracle_forward(const uint16_t *X, const uint16_t *phi, const uint16_t *F_out, int64_t B,
                    int n, int64_t C, double a_pre, double a_post, double a_res,
                    const double *bias, int iters, double *Y, double *r, double *H_pre,
                    double *H_post, double *H_res, double *F_pre, double *X_next)
{
    oracle_gemm_rms(X, phi, B, n, C, Y, r);
    oracle_coeffs(Y, r, a_pre, a_post, a_res, bias, iters, B, n, H_pre, H_post, H_res);
    oracle_pre_apply(X, H_pre, B, n, C, F_pre);
    oracle_post_res_apply(X, F_out, H_res, H_post, B, n, C, X_next);
}

/*
 * "Towards Free Normalization", §2: C = rmsnorm(A) @ B, where every row a of
 * A is scaled by rstd = 1 / sqrt(Σ_q a_q² / K + eps) before the product.
 * A [M][K] bf16, Bm [K][N] bf16 (the mathematical orientation), C [M][N].
 */
void oracle_rmsnorm_gemm(const uint16_t *A, const uint16_t *Bm, int64_t M, int64_t K, int64_t N,
                         double eps, double *Cout)
{
    double *row = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
    for (int64_t m = 0; m < M; ++m) {
        double ss = 0.0;
        for (int64_t q = 0; q < K; ++q) {
            const double a = oracle_bf16_to_f64(A[m * K + q]);
            ss += a * a;
        }
        const double rstd = 1.0 / sqrt(ss / (double)K + eps);
        for (int64_t q = 0; q < K; ++q) row[q] = oracle_bf16_to_f64(A[m * K + q]) * rstd;
        for (int64_t k = 0; k < N; ++k) {
            double acc = 0.0;
            for (int64_t q = 0; q < K; ++q) acc += row[q] * oracle_bf16_to_f64(Bm[q * N + k]);
            Cout[m * N + k] = acc;
        }
    }
    free(row);
}

/*
 * The page's optimised benchmark (§5) keeps the weight in fp32 (TF32 MMA) and
 * the other inputs in fp32 while X stays bf16.  These variants take φ and F_out
 * as doubles (exact widenings of fp32); the arithmetic is that of
 * oracle_gemm_rms and oracle_post_res_apply.
 */
void oracle_gemm_rms_f64phi(const uint16_t *X, const double *phi, int64_t B, int n, int64_t C,
                            double *Y, double *r)
{
    const int64_t K = (int64_t)n * C;
    const int N = n * n + 2 * n;
    for (int64_t b = 0; b < B; ++b) {
        double ss = 0.0;
        for (int64_t q = 0; q < K; ++q) {
            const double x = oracle_bf16_to_f64(X[b * K + q]);
            ss += x * x;
        }
        r[b] = sqrt(ss / (double)K);
        for (int k = 0; k < N; ++k) {
            double acc = 0.0;
            for (int64_t q = 0; q < K; ++q) acc += oracle_bf16_to_f64(X[b * K + q]) * phi[q * N + k];
            Y[b * N + k] = acc;
        }
    }
}

void oracle_post_res_apply_f64F(const uint16_t *X, const double *F_out, const double *H_res,
                                const double *H_post, int64_t B, int n, int64_t C,
                                double *X_next)
{
    const int64_t K = (int64_t)n * C;
    for (int64_t b = 0; b < B; ++b) {
        const double *h = H_res + b * n * n;
        for (int i = 0; i < n; ++i)
            for (int64_t c = 0; c < C; ++c) {
                double x_res = 0.0;
                for (int j = 0; j < n; ++j)
                    x_res += h[i * n + j] * oracle_bf16_to_f64(X[b * K + (int64_t)j * C + c]);
                X_next[b * K + (int64_t)i * C + c] = x_res + H_post[b * n + i] * F_out[b * C + c];
            }
    }
}

void oracle_forward_f64w(const uint16_t *X, const double *phi, const double *F_out, int64_t B,
                         int n, int64_t C, double a_pre, double a_post, double a_res,
                         const double *bias, int iters, double *Y, double *r, double *H_pre,
                         double *H_post, double *H_res, double *F_pre, double *X_next)
{
    oracle_gemm_rms_f64phi(X, phi, B, n, C, Y, r);
    oracle_coeffs(Y, r, a_pre, a_post, a_res, bias, iters, B, n, H_pre, H_post, H_res);
    oracle_pre_apply(X, H_pre, B, n, C, F_pre);
    oracle_post_res_apply_f64F(X, F_out, H_res, H_post, B, n, C, X_next);
}

/*
 * The page's first benchmark (§4) runs the path in fp8 e4m3.  e4m3 (the OCP
 * 8-bit format E4M3): sign, 4 exponent bits with bias 7, 3 mantissa bits; no
 * infinities, S.1111.111 is NaN; exponent field 0 holds subnormals m·2^-9.
 */
double oracle_e4m3_to_f64(uint8_t b)
{
    const double s = (b & 0x80) ? -1.0 : 1.0;
    const int e = (b >> 3) & 0xF, m = b & 7;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) return s * ldexp((double)m, -9);
    return s * ldexp(1.0 + m / 8.0, e - 7);
}

/* The steps of §2 on decoded (double) inputs; X [B][K], phi [K][N], F_out [B][C]. */
static void gemm_rms_f64(const double *X, const double *phi, int64_t B, int n, int64_t C,
                         double *Y, double *r)
{
    const int64_t K = (int64_t)n * C;
    const int N = n * n + 2 * n;
    for (int64_t b = 0; b < B; ++b) {
        double ss = 0.0;
        for (int64_t q = 0; q < K; ++q) ss += X[b * K + q] * X[b * K + q];
        r[b] = sqrt(ss / (double)K);
        for (int k = 0; k < N; ++k) {
            double acc = 0.0;
            for (int64_t q = 0; q < K; ++q) acc += X[b * K + q] * phi[q * N + k];
            Y[b * N + k] = acc;
        }
    }
}

static void apply_f64(const double *X, const double *F_out, const double *H_pre,
                      const double *H_post, const double *H_res, int64_t B, int n, int64_t C,
                      double *F_pre, double *X_next)
{
    const int64_t K = (int64_t)n * C;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t c = 0; c < C; ++c) {
            double f = 0.0;
            for (int i = 0; i < n; ++i) f += H_pre[b * n + i] * X[b * K + (int64_t)i * C + c];
            F_pre[b * C + c] = f;
            for (int i = 0; i < n; ++i) {
                double x_res = 0.0;
                for (int j = 0; j < n; ++j)
                    x_res += H_res[b * n * n + i * n + j] * X[b * K + (int64_t)j * C + c];
                X_next[b * K + (int64_t)i * C + c] = x_res + H_post[b * n + i] * F_out[b * C + c];
            }
        }
}

/* The whole forward with X, φ [K][N] and F_out given as e4m3 codes. */
void oracle_forward_e4m3(const uint8_t *X, const uint8_t *phi, const uint8_t *F_out, int64_t B,
                         int n, int64_t C, double a_pre, double a_post, double a_res,
                         const double *bias, int iters, double *Y, double *r, double *H_pre,
                         double *H_post, double *H_res, double *F_pre, double *X_next)
{
    const int64_t K = (int64_t)n * C;
    const int N = n * n + 2 * n;
    double *Xd = (double *)malloc((size_t)(B * K > 0 ? B * K : 1) * sizeof(double));
    double *Pd = (double *)malloc((size_t)(K * N > 0 ? K * N : 1) * sizeof(double));
    double *Fd = (double *)malloc((size_t)(B * C > 0 ? B * C : 1) * sizeof(double));
    for (int64_t i = 0; i < B * K; ++i) Xd[i] = oracle_e4m3_to_f64(X[i]);
    for (int64_t i = 0; i < K * N; ++i) Pd[i] = oracle_e4m3_to_f64(phi[i]);
    for (int64_t i = 0; i < B * C; ++i) Fd[i] = oracle_e4m3_to_f64(F_out[i]);
    gemm_rms_f64(Xd, Pd, B, n, C, Y, r);
    oracle_coeffs(Y, r, a_pre, a_post, a_res, bias, iters, B, n, H_pre, H_post, H_res);
    apply_f64(Xd, Fd, H_pre, H_post, H_res, B, n, C, F_pre, X_next);
    free(Xd);
    free(Pd);
    free(Fd);
}
