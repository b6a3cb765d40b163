// Step 4 of the mHC forward: the two bandwidth-bound apply kernels (page
// "mHC 算法分析 & cutile 高效实现", §2.5; fusion §3.4; §5.4 uses plain FMAs,
// not MMA, for the n×n mixing).
//
//   pre:       F_pre[b][c]     = Σ_i H_pre[b][i]·X[b][i][c]
//   post/res:  X_next[b][i][c] = Σ_j H_res[b][i][j]·X[b][j][c] + H_post[b][i]·F_out[b][c]
//
// A thread owns 8 consecutive channels c of one token: it reads them from all
// n streams with 128-bit loads, mixes in fp32 and writes 128-bit stores, so X
// is read once and every output written once, fully coalesced.  A block
// covers a run of channels of one token (blockIdx.y walks the tokens), and
// the token's coefficients are staged once per block in shared memory.
// Streaming cache hints (.cs) keep the single-use data from displacing L2.
//
// In place: X_next may equal X.  Every thread loads all its inputs before it
// stores, and the addresses it stores are exactly the ones it loaded, which
// no other thread touches; the accesses are volatile asm, kept in order.
#include <cuda_runtime.h>

#include <cstdint>

#include "mhc_internal.h"
#include "mix.cuh"
#include "ptx.cuh"

namespace mhc {
namespace {

constexpr int kMaxGridY = 65535;

template <int n>
__global__ void pre_apply_kernel(const uint16_t *__restrict__ X, const float *__restrict__ H_pre,
                                 int64_t B, int64_t C, uint16_t *__restrict__ F_pre)
{
    const int64_t C8 = C >> 3;
    const int64_t c8 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    ptx::pdl_wait();  // H_pre comes from the previous kernel
    ptx::pdl_trigger();
    for (int64_t b = blockIdx.y; b < B; b += gridDim.y) {
        float h[n];
#pragma unroll
        for (int i = 0; i < n; ++i) h[i] = __ldg(H_pre + b * n + i);
        if (c8 < C8) {
            const uint16_t *x = X + b * n * C + c8 * 8;
            uint4 xv[n];
#pragma unroll
            for (int i = 0; i < n; ++i) xv[i] = ptx::ld_stream_v4(x + i * C);
            ptx::st_stream_v4(F_pre + b * C + c8 * 8, pre_mix8<n>(h, xv));
        }
    }
}

// Up to n = 4 the kernel fits in 64 registers: 8 blocks of 128 threads per SM,
// enough loads in flight to reach copy bandwidth (measured 305 µs against 312 µs
// at 72 registers, B=16384, C=7168).  Wider n is held to 128 registers.
// Eight consecutive F_out values as fp32, from bf16 (one 128-bit load) or fp32
// (two) storage.
__device__ __forceinline__ void load_f8(const uint16_t *p, float (&f)[8])
{
    unpack8(ptx::ld_stream_v4(p), f);
}
__device__ __forceinline__ void load_f8(const float *p, float (&f)[8])
{
    const uint4 a = ptx::ld_stream_v4(p), b = ptx::ld_stream_v4(p + 4);
    f[0] = __uint_as_float(a.x); f[1] = __uint_as_float(a.y);
    f[2] = __uint_as_float(a.z); f[3] = __uint_as_float(a.w);
    f[4] = __uint_as_float(b.x); f[5] = __uint_as_float(b.y);
    f[6] = __uint_as_float(b.z); f[7] = __uint_as_float(b.w);
}

// FT: the element type of F_out, uint16_t (bf16) or float.
template <int n, typename FT>
__global__ void __launch_bounds__(256, n <= 4 ? 4 : 2)
post_res_apply_kernel(const uint16_t *X, const FT *__restrict__ F_out,
                                      const float *__restrict__ H_res,
                                      const float *__restrict__ H_post, int64_t B, int64_t C,
                                      uint16_t *X_next)
{
    __shared__ float hs[n * n + n];
    const int64_t C8 = C >> 3;
    const int64_t c8 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    ptx::pdl_wait();  // H_res and H_post come from earlier kernels
    ptx::pdl_trigger();
    for (int64_t b = blockIdx.y; b < B; b += gridDim.y) {
        // the token's X and F_out are requested (into L2, no registers held)
        // before its coefficients, so the two round trips overlap; wider n has
        // no registers to spare for the addresses under its 128-register cap
        if constexpr (n <= 4) {
            if (c8 < C8) {
                const uint16_t *x = X + b * n * C + c8 * 8;
#pragma unroll
                for (int j = 0; j < n; ++j) ptx::prefetch_l2(x + j * C);
                ptx::prefetch_l2(F_out + b * C + c8 * 8);
            }
        }
        __syncthreads();  // previous token's coefficients are no longer read
        for (int t = threadIdx.x; t < n * n + n; t += blockDim.x)
            hs[t] = t < n * n ? __ldg(H_res + b * n * n + t) : __ldg(H_post + b * n + (t - n * n));
        __syncthreads();
        if (c8 < C8) {
            const uint16_t *x = X + b * n * C + c8 * 8;
            uint4 xv[n];
#pragma unroll
            for (int j = 0; j < n; ++j) xv[j] = ptx::ld_stream_v4(x + j * C);
            float f[8];
            load_f8(F_out + b * C + c8 * 8, f);
            uint16_t *y = X_next + b * n * C + c8 * 8;
#pragma unroll
            for (int i = 0; i < n; ++i) ptx::st_stream_v4(y + i * C, post_mix8<n>(hs, i, xv, f));
        }
    }
}

// Threads per block: a power of two that divides C/8 when one exists (no idle
// lanes), otherwise 128.
int block_threads(int64_t C8)
{
    for (int t : {256, 128, 64, 32})
        if (C8 % t == 0) return t;
    return 128;
}

dim3 apply_grid(int64_t B, int64_t C8, int threads)
{
    const int64_t gx = (C8 + threads - 1) / threads;
    const int64_t gy = B < kMaxGridY ? B : kMaxGridY;
    return dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), 1);
}

template <typename FT>
cudaError_t launch_post_res(const uint16_t *X, const FT *F_out, const float *H_res,
                            const float *H_post, int64_t B, int n, int64_t C, uint16_t *X_next,
                            cudaStream_t stream)
{
    const int64_t C8 = C / 8;
    const int threads = block_threads(C8);
    const dim3 grid = apply_grid(B, C8, threads);
    switch (n) {
#define MHC_CASE(k)                                                                            \
    case k:                                                                                    \
        return launch_pdl(post_res_apply_kernel<k, FT>, grid, dim3(threads), 0, stream, X,     \
                          F_out, H_res, H_post, B, C, X_next);
        MHC_CASE(1) MHC_CASE(2) MHC_CASE(3) MHC_CASE(4) MHC_CASE(5) MHC_CASE(6) MHC_CASE(7)
        MHC_CASE(8)
#undef MHC_CASE
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_pre_apply(const uint16_t *X, const float *H_pre, int64_t B, int n, int64_t C,
                             uint16_t *F_pre, cudaStream_t stream)
{
    const int64_t C8 = C / 8;
    const int threads = block_threads(C8);
    const dim3 grid = apply_grid(B, C8, threads);
    switch (n) {
#define MHC_CASE(k) \
    case k: return launch_pdl(pre_apply_kernel<k>, grid, dim3(threads), 0, stream, X, H_pre, B, C, F_pre);
        MHC_CASE(1) MHC_CASE(2) MHC_CASE(3) MHC_CASE(4) MHC_CASE(5) MHC_CASE(6) MHC_CASE(7)
        MHC_CASE(8)
#undef MHC_CASE
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_post_res_apply(const uint16_t *X, const uint16_t *F_out, const float *H_res,
                                  const float *H_post, int64_t B, int n, int64_t C,
                                  uint16_t *X_next, cudaStream_t stream)
{
    return launch_post_res(X, F_out, H_res, H_post, B, n, C, X_next, stream);
}

cudaError_t launch_post_res_apply_f32(const uint16_t *X, const float *F_out, const float *H_res,
                                      const float *H_post, int64_t B, int n, int64_t C,
                                      uint16_t *X_next, cudaStream_t stream)
{
    return launch_post_res(X, F_out, H_res, H_post, B, n, C, X_next, stream);
}

}  // namespace mhc
