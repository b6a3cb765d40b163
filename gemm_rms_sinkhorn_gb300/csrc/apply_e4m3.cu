// Step 4 of the mHC forward on fp8 e4m3 activations (page "mHC 算法分析 &
// cutile 高效实现", §2.5; the e4m3 precision of its first benchmark, §4):
//
//   pre:       F_pre[b][c]     = Σ_i H_pre[b][i]·X[b][i][c]
//   post/res:  X_next[b][i][c] = Σ_j H_res[b][i][j]·X[b][j][c] + H_post[b][i]·F_out[b][c]
//
// X, F_out, F_pre and X_next are e4m3 codes.  A thread owns 16 consecutive
// channels of one token: one 128-bit load from each of the n streams, decoded
// once into f16x2 pairs (exact: e4m3 is a subset of f16, one instruction per
// two values), mixed with f16x2 FMAs, and encoded straight to e4m3 (round to
// nearest even, saturating to ±448) into one 128-bit store.  f16's 2^-11
// rounding is far below e4m3's 2^-4, and with |X|, |F_out| <= 448 and the
// coefficients of a normalised forward (H_pre < 1, H_post < 2, Sinkhorn rows
// and columns near 1) every partial sum stays far inside f16's ±65504; only
// an unnormalised H_res (iters = 0 on large logits) could leave it, and then
// the output saturates.  Conversions through fp32 would cost several times the
// instructions of the memory traffic.  As in apply.cu a block covers a run of
// channels of one token, with the token's coefficients in shared memory, and
// every thread loads all its inputs before it stores, so X_next may be X.
#include <cuda_runtime.h>

#include <cstdint>

#include "check.cuh"
#include "mhc_internal.h"
#include "ptx.cuh"

namespace mhc {
namespace {

constexpr int kMaxGridY = 65535;

// 16 codes -> 8 f16x2 (pair p holds channels 2p, 2p+1), and back.
__device__ __forceinline__ void decode16(const uint4 &v, uint32_t (&h)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        h[2 * q] = e4m3x2_to_f16x2(w[q]);
        h[2 * q + 1] = e4m3x2_to_f16x2(w[q] >> 16);
    }
}

__device__ __forceinline__ uint4 encode16(const uint32_t (&h)[8])
{
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        w[q] = f16x2_to_e4m3x2(h[2 * q]) | (f16x2_to_e4m3x2(h[2 * q + 1]) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// For n <= 4 each thread takes two tokens per iteration (b and b + gridDim.y)
// and issues both tokens' loads before any arithmetic: twice the bytes in
// flight of one token at a time, which these kernels' register counts
// otherwise cap (measured 119 -> 81 µs and 174 -> 158 µs at B=16384, C=7168).
// Wider n has no registers for a second token (n = 8 measured slower with it).
template <int n>
constexpr int kTokens = n <= 4 ? 2 : 1;

template <int n>
__global__ void pre_apply_e4m3_kernel(const uint8_t *__restrict__ X,
                                      const float *__restrict__ H_pre, int64_t B, int64_t C,
                                      uint8_t *__restrict__ F_pre)
{
    const int64_t C16 = C >> 4;
    const int64_t c16 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    ptx::pdl_wait();
    ptx::pdl_trigger();
    if (c16 >= C16 || !in_range(201, c16 * 16, 16, C)) return;
    constexpr int kT = kTokens<n>;
    const int64_t step = static_cast<int64_t>(gridDim.y);
    for (int64_t b0 = blockIdx.y; b0 < B; b0 += kT * step) {
        int64_t bb[kT];
#pragma unroll
        for (int u = 0; u < kT; ++u) bb[u] = b0 + u * step;
        uint4 xv[kT][n];
#pragma unroll
        for (int u = 0; u < kT; ++u)
            if (bb[u] < B && in_range(202, bb[u], 1, B)) {
                const uint8_t *x = X + bb[u] * n * C + c16 * 16;
#pragma unroll
                for (int i = 0; i < n; ++i) xv[u][i] = ptx::ld_stream_v4(x + i * C);
            }
#pragma unroll
        for (int u = 0; u < kT; ++u) {
            if (bb[u] >= B || !in_range(203, bb[u], 1, B)) break;
            uint32_t acc[8], t[8];
#pragma unroll
            for (int p = 0; p < 8; ++p) acc[p] = 0u;  // +0, +0
#pragma unroll
            for (int i = 0; i < n; ++i) {
                const uint32_t h = f16x2_splat(__ldg(H_pre + bb[u] * n + i));
                decode16(xv[u][i], t);
#pragma unroll
                for (int p = 0; p < 8; ++p) acc[p] = hfma2(h, t[p], acc[p]);
            }
            ptx::st_stream_v4(F_pre + bb[u] * C + c16 * 16, encode16(acc));
        }
    }
}

template <int n>
__global__ void __launch_bounds__(256)
post_res_apply_e4m3_kernel(const uint8_t *X, const uint8_t *__restrict__ F_out,
                           const float *__restrict__ H_res, const float *__restrict__ H_post,
                           int64_t B, int64_t C, uint8_t *X_next)
{
    constexpr int kH = n * n + n;
    constexpr int kT = kTokens<n>;
    __shared__ uint32_t hs[kT][kH];  // f16x2 (v, v): H_res row-major, then H_post, per token
    const int64_t C16 = C >> 4;
    const int64_t c16 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const bool active = c16 < C16 && in_range(211, c16 * 16, 16, C);
    ptx::pdl_wait();
    ptx::pdl_trigger();
    const int64_t step = static_cast<int64_t>(gridDim.y);
    for (int64_t b0 = blockIdx.y; b0 < B; b0 += kT * step) {
        int64_t bb[kT];
#pragma unroll
        for (int u = 0; u < kT; ++u) bb[u] = b0 + u * step;
        bool tok[kT];
#pragma unroll
        for (int u = 0; u < kT; ++u) tok[u] = bb[u] < B && in_range(212, bb[u], 1, B);
        uint4 xv[kT][n], fv[kT];
        if constexpr (kT > 1) {
            // all tokens' loads first, in flight while the coefficients are staged
            if (active) {
#pragma unroll
                for (int u = 0; u < kT; ++u)
                    if (tok[u]) {
                        const uint8_t *x = X + bb[u] * n * C + c16 * 16;
#pragma unroll
                        for (int j = 0; j < n; ++j) xv[u][j] = ptx::ld_stream_v4(x + j * C);
                        fv[u] = ptx::ld_stream_v4(F_out + bb[u] * C + c16 * 16);
                    }
            }
        }
        __syncthreads();  // the previous tokens' coefficients are no longer read
        for (int t = threadIdx.x; t < kT * kH; t += blockDim.x) {
            const int u = t / kH, k = t - u * kH;
            if (bb[u] < B && in_range(213, bb[u], 1, B))
                hs[u][k] = f16x2_splat(k < n * n ? __ldg(H_res + bb[u] * n * n + k)
                                                 : __ldg(H_post + bb[u] * n + (k - n * n)));
        }
        __syncthreads();
        if (!active) continue;
#pragma unroll
        for (int u = 0; u < kT; ++u) {
            if (!tok[u]) break;
            uint32_t xh[n][8], fh[8];
            if constexpr (kT > 1) {
#pragma unroll
                for (int j = 0; j < n; ++j) decode16(xv[u][j], xh[j]);
                decode16(fv[u], fh);
            } else {
                // one token: load and decode here, no registers held across the syncs
                const uint8_t *x = X + bb[u] * n * C + c16 * 16;
#pragma unroll
                for (int j = 0; j < n; ++j) decode16(ptx::ld_stream_v4(x + j * C), xh[j]);
                decode16(ptx::ld_stream_v4(F_out + bb[u] * C + c16 * 16), fh);
            }
            uint8_t *y = X_next + bb[u] * n * C + c16 * 16;
#pragma unroll
            for (int i = 0; i < n; ++i) {
                uint32_t acc[8];
#pragma unroll
                for (int p = 0; p < 8; ++p) acc[p] = 0u;
#pragma unroll
                for (int j = 0; j < n; ++j)
#pragma unroll
                    for (int p = 0; p < 8; ++p) acc[p] = hfma2(hs[u][i * n + j], xh[j][p], acc[p]);
#pragma unroll
                for (int p = 0; p < 8; ++p) acc[p] = hfma2(hs[u][n * n + i], fh[p], acc[p]);
                ptx::st_stream_v4(y + i * C, encode16(acc));
            }
        }
    }
}

int block_threads16(int64_t C16)
{
    for (int t : {256, 128, 64, 32})
        if (C16 % t == 0) return t;
    return 128;
}

// kT tokens per block row and iteration.
dim3 grid16(int64_t B, int64_t C16, int threads, int kT)
{
    const int64_t gx = (C16 + threads - 1) / threads;
    const int64_t rows = (B + kT - 1) / kT;
    const int64_t gy = rows < kMaxGridY ? rows : kMaxGridY;
    return dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), 1);
}

}  // namespace

cudaError_t launch_pre_apply_e4m3(const uint8_t *X, const float *H_pre, int64_t B, int n,
                                  int64_t C, uint8_t *F_pre, cudaStream_t stream)
{
    const int64_t C16 = C / 16;
    const int threads = block_threads16(C16);
    switch (n) {
#define MHC_CASE(k)                                                                               \
    case k:                                                                                       \
        return launch_pdl(pre_apply_e4m3_kernel<k>, grid16(B, C16, threads, kTokens<k>),          \
                          dim3(threads), 0, stream, X, H_pre, B, C, F_pre);
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
    switch (n) {
#define MHC_CASE(k)                                                                               \
    case k:                                                                                       \
        return launch_pdl(post_res_apply_e4m3_kernel<k>, grid16(B, C16, threads, kTokens<k>),     \
                          dim3(threads), 0, stream, X, F_out, H_res, H_post, B, C, X_next);
        MHC_CASE(1) MHC_CASE(2) MHC_CASE(3) MHC_CASE(4) MHC_CASE(5) MHC_CASE(6) MHC_CASE(7)
        MHC_CASE(8)
#undef MHC_CASE
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace mhc
