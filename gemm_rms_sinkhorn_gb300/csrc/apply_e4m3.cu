// Step 4 of the mHC forward on fp8 e4m3 activations (page "mHC 算法分析 &
// cutile 高效实现", §2.5; the e4m3 precision of its first benchmark, §4):
//
//   pre:       F_pre[b][c]     = Σ_i H_pre[b][i]·X[b][i][c]
//   post/res:  X_next[b][i][c] = Σ_j H_res[b][i][j]·X[b][j][c] + H_post[b][i]·F_out[b][c]
//
// X, F_out, F_pre and X_next are e4m3 codes.  A thread owns 16 consecutive
// channels of one token: one 128-bit load from each of the n streams, exact
// decoding to fp32, fp32 FMAs, and e4m3 encoding (round to nearest even,
// saturating to ±448) into one 128-bit store.  As in apply.cu a block covers
// a run of channels of one token, with the token's coefficients in shared
// memory, and every thread loads all its inputs before it stores, so
// X_next may be X.
#include <cuda_runtime.h>

#include <cstdint>

#include "mhc_internal.h"
#include "ptx.cuh"

namespace mhc {
namespace {

constexpr int kMaxGridY = 65535;

__device__ __forceinline__ void decode16(const uint4 &v, float (&f)[16])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        e4m3x2_to_f32(w[h], f[4 * h], f[4 * h + 1]);
        e4m3x2_to_f32(w[h] >> 16, f[4 * h + 2], f[4 * h + 3]);
    }
}

__device__ __forceinline__ uint4 encode16(const float (&f)[16])
{
    uint32_t w[4];
#pragma unroll
    for (int h = 0; h < 4; ++h)
        w[h] = f32x2_to_e4m3(f[4 * h], f[4 * h + 1]) | (f32x2_to_e4m3(f[4 * h + 2], f[4 * h + 3]) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int n>
__global__ void pre_apply_e4m3_kernel(const uint8_t *__restrict__ X,
                                      const float *__restrict__ H_pre, int64_t B, int64_t C,
                                      uint8_t *__restrict__ F_pre)
{
    const int64_t C16 = C >> 4;
    const int64_t c16 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    ptx::pdl_wait();
    ptx::pdl_trigger();
    for (int64_t b = blockIdx.y; b < B; b += gridDim.y) {
        if (c16 >= C16) continue;
        float h[n];
#pragma unroll
        for (int i = 0; i < n; ++i) h[i] = __ldg(H_pre + b * n + i);
        const uint8_t *x = X + b * n * C + c16 * 16;
        uint4 xv[n];
#pragma unroll
        for (int i = 0; i < n; ++i) xv[i] = ptx::ld_stream_v4(x + i * C);
        float acc[16], t[16];
        decode16(xv[0], t);
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e] = h[0] * t[e];
#pragma unroll
        for (int i = 1; i < n; ++i) {
            decode16(xv[i], t);
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[e] = fmaf(h[i], t[e], acc[e]);
        }
        ptx::st_stream_v4(F_pre + b * C + c16 * 16, encode16(acc));
    }
}

template <int n>
__global__ void __launch_bounds__(256)
post_res_apply_e4m3_kernel(const uint8_t *X, const uint8_t *__restrict__ F_out,
                           const float *__restrict__ H_res, const float *__restrict__ H_post,
                           int64_t B, int64_t C, uint8_t *X_next)
{
    __shared__ float hs[n * n + n];
    const int64_t C16 = C >> 4;
    const int64_t c16 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    ptx::pdl_wait();
    ptx::pdl_trigger();
    for (int64_t b = blockIdx.y; b < B; b += gridDim.y) {
        __syncthreads();  // the previous token's coefficients are no longer read
        for (int t = threadIdx.x; t < n * n + n; t += blockDim.x)
            hs[t] = t < n * n ? __ldg(H_res + b * n * n + t) : __ldg(H_post + b * n + (t - n * n));
        __syncthreads();
        if (c16 >= C16) continue;
        const uint8_t *x = X + b * n * C + c16 * 16;
        uint4 xv[n];
#pragma unroll
        for (int j = 0; j < n; ++j) xv[j] = ptx::ld_stream_v4(x + j * C);
        float f[16];
        decode16(ptx::ld_stream_v4(F_out + b * C + c16 * 16), f);
        uint8_t *y = X_next + b * n * C + c16 * 16;
#pragma unroll 1
        for (int i = 0; i < n; ++i) {
            float acc[16], t[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[e] = 0.f;
#pragma unroll
            for (int j = 0; j < n; ++j) {
                const float hij = hs[i * n + j];
                decode16(xv[j], t);
#pragma unroll
                for (int e = 0; e < 16; ++e) acc[e] = fmaf(hij, t[e], acc[e]);
            }
            const float hq = hs[n * n + i];
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[e] = fmaf(hq, f[e], acc[e]);
            ptx::st_stream_v4(y + i * C, encode16(acc));
        }
    }
}

int block_threads16(int64_t C16)
{
    for (int t : {256, 128, 64, 32})
        if (C16 % t == 0) return t;
    return 128;
}

dim3 grid16(int64_t B, int64_t C16, int threads)
{
    const int64_t gx = (C16 + threads - 1) / threads;
    const int64_t gy = B < kMaxGridY ? B : kMaxGridY;
    return dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), 1);
}

}  // namespace

cudaError_t launch_pre_apply_e4m3(const uint8_t *X, const float *H_pre, int64_t B, int n,
                                  int64_t C, uint8_t *F_pre, cudaStream_t stream)
{
    const int64_t C16 = C / 16;
    const int threads = block_threads16(C16);
    const dim3 grid = grid16(B, C16, threads);
    switch (n) {
#define MHC_CASE(k)                                                                               \
    case k:                                                                                       \
        return launch_pdl(pre_apply_e4m3_kernel<k>, grid, dim3(threads), 0, stream, X, H_pre, B,  \
                          C, F_pre);
        MHC_CASE(1) MHC_CASE(2) MHC_CASE(3) MHC_CASE(4) MHC_CASE(5) MHC_CASE(6) MHC_CASE(7)
        MHC_CASE(8)
#undef MHC_CASE
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_post_res_apply_e4m3(const uint8_t *X, const uint8_t *F_out, const float *H_res,
                                       const float *H_post, int64_t B, int n, int64_t C,
                                       uint8_t *X_next, cudaStream_t stream)
{
    const int64_t C16 = C / 16;
    const int threads = block_threads16(C16);
    const dim3 grid = grid16(B, C16, threads);
    switch (n) {
#define MHC_CASE(k)                                                                               \
    case k:                                                                                       \
        return launch_pdl(post_res_apply_e4m3_kernel<k>, grid, dim3(threads), 0, stream, X, F_out, \
                          H_res, H_post, B, C, X_next);
        MHC_CASE(1) MHC_CASE(2) MHC_CASE(3) MHC_CASE(4) MHC_CASE(5) MHC_CASE(6) MHC_CASE(7)
        MHC_CASE(8)
#undef MHC_CASE
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace mhc
