// Steps 2–3 of the mHC forward: scale / α / bias, the sigmoid constraints and
// the Sinkhorn–Knopp projection, fused into one kernel (page "mHC 算法分析 &
// cutile 高效实现", §2.3, §2.4; fusions §3.2 and §3.3; §5.3 keeps the n×n
// block in registers).
//
//   H̃ = α_seg·Y/r + b;  H_pre = σ(H̃_pre);  H_post = 2σ(H̃_post)
//   H_res = exp(H̃_res), then `iters` × (rows /= row sums; columns /= column sums)
//
// One thread owns one token: its n×n block lives in registers for all
// iterations.  Y rows are staged through shared memory so global loads and
// stores stay coalesced; the N = n²+2n outputs of a token overwrite its own
// Y row in shared memory and leave in three coalesced streams.
//
// Before the first row normalisation each row is shifted by its maximum:
// exp(h - m)/Σ exp(h - m) = exp(h)/Σ exp(h), so every iterate from the first
// row step on is unchanged in exact arithmetic while exp cannot overflow.
// With iters = 0 the raw exp(H̃_res) is returned and no shift is applied.
#include <cuda_runtime.h>

#include <cstdint>

#include "mhc_internal.h"

namespace mhc {
namespace {

constexpr int kTokensPerBlock = 128;

template <int n>
__global__ void __launch_bounds__(kTokensPerBlock)
coeffs_kernel(const float *__restrict__ Y, const float *__restrict__ r, float a_pre, float a_post,
              float a_res, const float *__restrict__ bias, int iters, int64_t B,
              float *__restrict__ H_pre, float *__restrict__ H_post, float *__restrict__ H_res)
{
    constexpr int N = n * n + 2 * n;
    __shared__ float rows_s[kTokensPerBlock * N];
    __shared__ float bias_s[N];

    const int64_t b0 = static_cast<int64_t>(blockIdx.x) * kTokensPerBlock;
    const int rows = static_cast<int>(B - b0 < kTokensPerBlock ? B - b0 : kTokensPerBlock);
    for (int i = threadIdx.x; i < rows * N; i += kTokensPerBlock) rows_s[i] = Y[b0 * N + i];
    if (threadIdx.x < N) bias_s[threadIdx.x] = bias[threadIdx.x];
    __syncthreads();

    if (threadIdx.x < rows) {
        float *h = rows_s + threadIdx.x * N;
        const float rb = r[b0 + threadIdx.x];
        // §2.3 + §2.4 for the pre and post segments
#pragma unroll
        for (int i = 0; i < n; ++i) {
            const float tp = a_pre * h[i] / rb + bias_s[i];
            const float tq = a_post * h[n + i] / rb + bias_s[n + i];
            h[i] = 1.0f / (1.0f + expf(-tp));
            h[n + i] = 2.0f / (1.0f + expf(-tq));
        }
        // §2.4 Sinkhorn–Knopp on the res segment
        float m[n][n];
#pragma unroll
        for (int i = 0; i < n; ++i)
#pragma unroll
            for (int j = 0; j < n; ++j)
                m[i][j] = a_res * h[2 * n + i * n + j] / rb + bias_s[2 * n + i * n + j];
        if (iters > 0) {
#pragma unroll
            for (int i = 0; i < n; ++i) {
                float mx = m[i][0];
#pragma unroll
                for (int j = 1; j < n; ++j) mx = fmaxf(mx, m[i][j]);
#pragma unroll
                for (int j = 0; j < n; ++j) m[i][j] = expf(m[i][j] - mx);
            }
        } else {
#pragma unroll
            for (int i = 0; i < n; ++i)
#pragma unroll
                for (int j = 0; j < n; ++j) m[i][j] = expf(m[i][j]);
        }
        for (int t = 0; t < iters; ++t) {
#pragma unroll
            for (int i = 0; i < n; ++i) {
                float s = 0.f;
#pragma unroll
                for (int j = 0; j < n; ++j) s += m[i][j];
#pragma unroll
                for (int j = 0; j < n; ++j) m[i][j] = m[i][j] / s;
            }
#pragma unroll
            for (int j = 0; j < n; ++j) {
                float s = 0.f;
#pragma unroll
                for (int i = 0; i < n; ++i) s += m[i][j];
#pragma unroll
                for (int i = 0; i < n; ++i) m[i][j] = m[i][j] / s;
            }
        }
#pragma unroll
        for (int i = 0; i < n; ++i)
#pragma unroll
            for (int j = 0; j < n; ++j) h[2 * n + i * n + j] = m[i][j];
    }
    __syncthreads();

    for (int e = threadIdx.x; e < rows * n; e += kTokensPerBlock) {
        const int t = e / n, i = e - t * n;
        H_pre[b0 * n + e] = rows_s[t * N + i];
        H_post[b0 * n + e] = rows_s[t * N + n + i];
    }
    for (int e = threadIdx.x; e < rows * n * n; e += kTokensPerBlock) {
        const int t = e / (n * n), ij = e - t * (n * n);
        H_res[b0 * n * n + e] = rows_s[t * N + 2 * n + ij];
    }
}

template <int n>
cudaError_t launch_n(const float *Y, const float *r, float a_pre, float a_post, float a_res,
                     const float *bias, int iters, int64_t B, float *H_pre, float *H_post,
                     float *H_res, cudaStream_t stream)
{
    const int64_t blocks = (B + kTokensPerBlock - 1) / kTokensPerBlock;
    coeffs_kernel<n><<<static_cast<unsigned>(blocks), kTokensPerBlock, 0, stream>>>(
        Y, r, a_pre, a_post, a_res, bias, iters, B, H_pre, H_post, H_res);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_coeffs(const float *Y, const float *r, float a_pre, float a_post, float a_res,
                          const float *bias, int iters, int64_t B, int n, float *H_pre,
                          float *H_post, float *H_res, cudaStream_t stream)
{
    switch (n) {
#define MHC_CASE(k) \
    case k: return launch_n<k>(Y, r, a_pre, a_post, a_res, bias, iters, B, H_pre, H_post, H_res, stream);
        MHC_CASE(1) MHC_CASE(2) MHC_CASE(3) MHC_CASE(4) MHC_CASE(5) MHC_CASE(6) MHC_CASE(7)
        MHC_CASE(8)
#undef MHC_CASE
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace mhc
