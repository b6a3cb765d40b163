// Steps 2–3 of the mHC forward: scale / α / bias, the sigmoid constraints and
// the Sinkhorn–Knopp projection, fused into one kernel (page "mHC 算法分析 &
// cutile 高效实现", §2.3, §2.4; fusions §3.2 and §3.3; §5.3 keeps the n×n
// block in registers).
//
//   H̃ = α_seg·Y/r + b;  H_pre = σ(H̃_pre);  H_post = 2σ(H̃_post)
//   H_res = exp(H̃_res), then `iters` × (rows /= row sums; columns /= column sums)
//
// A token is handled by a group of n consecutive lanes of a warp; lane i of
// the group owns row i of the n×n block (in registers) and entry i of the pre
// and post segments.  Row sums are lane-local; column sums are a shuffle
// reduction across the group that every lane evaluates in the same order, so
// all lanes divide a column by the identical sum.  Each normalisation takes
// one correctly rounded reciprocal per sum and multiplies by it (at most one
// rounding away from a true division).  Spreading a token over n lanes gives
// the serial iteration n times more warps to hide its latency.
//
// Before the first row normalisation each row is shifted by its maximum:
// exp(h - m)/Σ exp(h - m) = exp(h)/Σ exp(h), so every iterate from the first
// row step on is unchanged in exact arithmetic while exp cannot overflow.
// With iters = 0 the raw exp(H̃_res) is returned and no shift is applied.
#include <cuda_runtime.h>

#include <cstdint>

#include "mhc_internal.h"
#include "ptx.cuh"

namespace mhc {
namespace {

constexpr int kThreads = 128;

// Sum over the n lanes of a token group of v, identical on every lane.
template <int n>
__device__ __forceinline__ float group_sum(float v, int base, unsigned mask)
{
    if constexpr ((n & (n - 1)) == 0) {
        // butterfly: a + b == b + a exactly, so every lane ends with the same value
#pragma unroll
        for (int off = 1; off < n; off <<= 1) v += __shfl_xor_sync(mask, v, off);
        return v;
    } else {
        float s = __shfl_sync(mask, v, base);
#pragma unroll
        for (int k = 1; k < n; ++k) s += __shfl_sync(mask, v, base + k);
        return s;
    }
}

template <int n>
__global__ void __launch_bounds__(kThreads)
coeffs_kernel(const float *__restrict__ Y, const float *__restrict__ r, float a_pre, float a_post,
              float a_res, const float *__restrict__ bias, int iters, int64_t B,
              float *__restrict__ H_pre, float *__restrict__ H_post, float *__restrict__ H_res)
{
    constexpr int N = n * n + 2 * n;
    constexpr int kGroups = 32 / n;  // tokens per warp
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int g = lane / n;          // token group within the warp
    const int i = lane - g * n;      // row owned by this lane
    const int base = g * n;
    // lanes of whole groups take part in the shuffles; the spare lanes
    // (32 mod n of them) sit out
    const unsigned mask = kGroups * n == 32 ? 0xFFFFFFFFu : ((1u << (kGroups * n)) - 1u);
    if (g >= kGroups) return;
    ptx::pdl_wait();  // Y and r come from the previous kernel
    ptx::pdl_trigger();

    const int64_t t = (static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + warp) * kGroups + g;
    const bool valid = t < B;
    const int64_t tt = valid ? t : B - 1;  // idle groups mirror the last token, store nothing
    const float *y = Y + tt * N;
    const float rb = __ldg(r + tt);

    // §2.3 + §2.4, pre and post entries i
    const float tp = a_pre * __ldg(y + i) / rb + __ldg(bias + i);
    const float tq = a_post * __ldg(y + n + i) / rb + __ldg(bias + n + i);
    const float hp = 1.0f / (1.0f + expf(-tp));
    const float hq = 2.0f / (1.0f + expf(-tq));

    // §2.4 Sinkhorn–Knopp, row i of the res block
    float m[n];
#pragma unroll
    for (int j = 0; j < n; ++j)
        m[j] = a_res * __ldg(y + 2 * n + i * n + j) / rb + __ldg(bias + 2 * n + i * n + j);
    if (iters > 0) {
        float mx = m[0];
#pragma unroll
        for (int j = 1; j < n; ++j) mx = fmaxf(mx, m[j]);
#pragma unroll
        for (int j = 0; j < n; ++j) m[j] = expf(m[j] - mx);
    } else {
#pragma unroll
        for (int j = 0; j < n; ++j) m[j] = expf(m[j]);
    }
    for (int it = 0; it < iters; ++it) {
        float s = m[0];
#pragma unroll
        for (int j = 1; j < n; ++j) s += m[j];
        const float inv = __frcp_rn(s);
#pragma unroll
        for (int j = 0; j < n; ++j) m[j] *= inv;
#pragma unroll
        for (int j = 0; j < n; ++j) m[j] *= __frcp_rn(group_sum<n>(m[j], base, mask));
    }

    if (valid) {
        H_pre[t * n + i] = hp;
        H_post[t * n + i] = hq;
        float *o = H_res + t * n * n + i * n;
#pragma unroll
        for (int j = 0; j < n; ++j) o[j] = m[j];
    }
}

template <int n>
cudaError_t launch_n(const float *Y, const float *r, float a_pre, float a_post, float a_res,
                     const float *bias, int iters, int64_t B, float *H_pre, float *H_post,
                     float *H_res, cudaStream_t stream)
{
    constexpr int64_t tokens_per_block = (kThreads / 32) * (32 / n);
    const int64_t blocks = (B + tokens_per_block - 1) / tokens_per_block;
    return launch_pdl(coeffs_kernel<n>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0,
                      stream, Y, r, a_pre, a_post, a_res, bias, iters, B, H_pre, H_post, H_res);
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
