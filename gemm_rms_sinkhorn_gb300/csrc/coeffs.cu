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
#include "mix.cuh"
#include "ptx.cuh"

namespace mhc {
namespace {

constexpr int kThreads = 128;

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
    // lanes of whole groups take part in the shuffles; the spare lanes
    // (32 mod n of them) sit out
    const unsigned mask = kGroups * n == 32 ? 0xFFFFFFFFu : ((1u << (kGroups * n)) - 1u);
    if (g >= kGroups) return;
    ptx::pdl_wait();  // Y and r come from the previous kernel
    ptx::pdl_trigger();

    const int64_t t = (static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + warp) * kGroups + g;
    const bool valid = t < B;
    const int64_t tt = valid ? t : B - 1;  // idle groups mirror the last token, store nothing
    float hp, hq, m[n];
    coeff_lane<n>(Y + tt * N, __ldg(r + tt), bias, a_pre, a_post, a_res, iters, i, g * n, mask, hp,
                  hq, m);
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
