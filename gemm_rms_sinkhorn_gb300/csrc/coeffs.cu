// Steps 2–3 of the mHC forward: scale / α / bias, the sigmoid constraints and
// the Sinkhorn–Knopp projection, fused into one kernel (page "mHC 算法分析 &
// cutile 高效实现", §2.3, §2.4; fusions §3.2 and §3.3; §5.3 keeps the n×n
// block in registers).
//
//   H̃ = α_seg·Y/r + b;  H_pre = σ(H̃_pre);  H_post = 2σ(H̃_post)
//   H_res = exp(H̃_res), then `iters` × (rows /= row sums; columns /= column sums)
//
// One thread per token holds the whole n×n block in registers (token_coeffs),
// so the iteration needs no communication between threads and its latency is
// one thread's dependency chain: the n row (then column) sums of a step are
// independent and overlap.  Y rows are read with 128-bit loads when N keeps
// them 16-byte aligned (n even).
#include <cuda_runtime.h>

#include <cstdint>

#include "check.cuh"
#include "mhc_internal.h"
#include "mix.cuh"
#include "ptx.cuh"

namespace mhc {
namespace {

constexpr int kThreads = 64;  // small blocks spread a mid-size batch over more SMs

template <int n>
__global__ void __launch_bounds__(kThreads)
coeffs_kernel(const float *__restrict__ Y, const float *__restrict__ r, float a_pre, float a_post,
              float a_res, const float *__restrict__ bias, int iters, int64_t B,
              float *__restrict__ H_pre, float *__restrict__ H_post, float *__restrict__ H_res)
{
    constexpr int N = n * n + 2 * n;
    ptx::pdl_wait();  // Y and r come from the previous kernel
    ptx::pdl_trigger();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; t < B;
         t += stride) {
        if (!in_range(301, t, 1, B)) break;  // Y, r and the three outputs: row t
        float y[N];
        if constexpr (N % 4 == 0) {
            const float4 *src = reinterpret_cast<const float4 *>(Y + t * N);
#pragma unroll
            for (int k = 0; k < N / 4; ++k) {
                const float4 v = __ldg(src + k);
                y[4 * k] = v.x; y[4 * k + 1] = v.y; y[4 * k + 2] = v.z; y[4 * k + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int k = 0; k < N; ++k) y[k] = __ldg(Y + t * N + k);
        }
        float hp[n], hq[n], m[n][n];
        token_coeffs<n>(y, __ldg(r + t), bias, a_pre, a_post, a_res, iters, hp, hq, m);
        store_token_coeffs<n>(t, hp, hq, m, H_pre, H_post, H_res);
    }
}

template <int n>
cudaError_t launch_n(const float *Y, const float *r, float a_pre, float a_post, float a_res,
                     const float *bias, int iters, int64_t B, float *H_pre, float *H_post,
                     float *H_res, cudaStream_t stream)
{
    const int64_t need = (B + kThreads - 1) / kThreads;
    const int64_t blocks = need < (int64_t{1} << 20) ? need : (int64_t{1} << 20);
    return launch_pdl(coeffs_kernel<n>, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0,
                      stream, Y, r, a_pre, a_post, a_res, bias, iters, B, H_pre, H_post, H_res);
}

__global__ void recip_kernel(const float *__restrict__ in, float *__restrict__ out, int64_t count)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
         i += stride)
        if (in_range(302, i, 1, count)) out[i] = recip_approx(in[i]);
}

}  // namespace

cudaError_t launch_recip(const float *in, float *out, int64_t count, cudaStream_t stream)
{
    const int64_t need = (count + 255) / 256;
    const int blocks = static_cast<int>(need < 4096 ? need : 4096);
    recip_kernel<<<blocks, 256, 0, stream>>>(in, out, count);
    return cudaGetLastError();
}

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
