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
// Wide n (5..8) runs a set number of waves' worth of blocks instead, each
// walking the tokens b, b + gridDim.y, ...: while it mixes one token, the
// next token's coefficients are already on their way (into shared memory by
// cp.async for post/res, into registers for pre), and for post/res its X and
// F_out into L2 (prefetch), so a token does not wait for a coefficient round
// trip before its DRAM round trip.  Measured at n = 8, C = 4096: against one
// token per block, post/res 11-14 % faster with the prefetch (B = 2048..8192).
// Its walks are best at about 6 tokens: at B = 8192, 178 µs at 27 tokens a
// walk, 172 at 4-7, 176 at 2, 193 at 1 (nothing left to hide the next token
// behind); 2-5 % faster than a fixed two waves at B = 3072..16384, the same
// below.  Pre is fastest at one token per block (95 µs at B = 8192 with walks
// of 7 tokens, 90-91 µs with 1-2), so it takes 32 waves.
//
// In place: X_next may equal X.  Every thread loads all its inputs before it
// stores, and the addresses it stores are exactly the ones it loaded, which
// no other thread touches; the accesses are volatile asm, kept in order.  A
// prefetch of the next token's lines only moves them into L2.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "check.cuh"
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
        if (!in_range(101, b, 1, B)) continue;
        float h[n];
#pragma unroll
        for (int i = 0; i < n; ++i) h[i] = __ldg(H_pre + b * n + i);
        if (c8 < C8 && in_range(102, c8 * 8, 8, C)) {
            const uint16_t *x = X + b * n * C + c8 * 8;
            uint4 xv[n];
#pragma unroll
            for (int i = 0; i < n; ++i) xv[i] = ptx::ld_stream_v4(x + i * C);
            ptx::st_stream_v4(F_pre + b * C + c8 * 8, pre_mix8<n>(h, xv));
        }
    }
}

// Wide n: the blocks walk the tokens; the next token's H_pre is loaded into
// registers before this token is mixed.
template <int n>
__global__ void __launch_bounds__(256, 4)
pre_apply_wide_kernel(const uint16_t *__restrict__ X, const float *__restrict__ H_pre, int64_t B,
                      int64_t C, uint16_t *__restrict__ F_pre)
{
    const int64_t C8 = C >> 3;
    const int64_t c8 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const bool active = c8 < C8;
    ptx::pdl_wait();  // H_pre comes from the previous kernel
    ptx::pdl_trigger();
    int64_t b = blockIdx.y;
    float h[n];
#pragma unroll
    for (int i = 0; i < n; ++i) h[i] = b < B ? __ldg(H_pre + b * n + i) : 0.f;
    for (; b < B; b += gridDim.y) {
        const int64_t bn = b + gridDim.y;
        const uint16_t *x = X + b * n * C + c8 * 8;
        uint4 xv[n];
        if (!in_range(103, b, 1, B)) break;
        const bool ok = active && in_range(104, c8 * 8, 8, C);
        if (ok) {
#pragma unroll
            for (int i = 0; i < n; ++i) xv[i] = ptx::ld_stream_v4(x + i * C);
        }
        float hn[n];
#pragma unroll
        for (int i = 0; i < n; ++i) hn[i] = bn < B ? __ldg(H_pre + bn * n + i) : 0.f;
        if (ok) ptx::st_stream_v4(F_pre + b * C + c8 * 8, pre_mix8<n>(h, xv));
#pragma unroll
        for (int i = 0; i < n; ++i) h[i] = hn[i];
    }
}

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

// n <= 4.  FT: the element type of F_out, uint16_t (bf16) or float.  The
// kernel fits in 64 registers: 8 blocks of 128 threads per SM, enough loads in
// flight to reach copy bandwidth (measured 305 µs against 312 µs at 72
// registers, B=16384, C=7168).
template <int n, typename FT>
__global__ void __launch_bounds__(256, 4)
post_res_apply_kernel(const uint16_t *X, const FT *__restrict__ F_out,
                      const float *__restrict__ H_res, const float *__restrict__ H_post,
                      int64_t B, int64_t C, uint16_t *X_next)
{
    static_assert(n <= 4, "wide n takes post_res_apply_wide_kernel");
    __shared__ float hs[n * n + n];
    const int64_t C8 = C >> 3;
    const int64_t c8 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    ptx::pdl_wait();  // H_res and H_post come from earlier kernels
    ptx::pdl_trigger();
    // the last tokens first: pre_apply, which runs just before in mhc_forward,
    // read them last, so part of their X is still in L2
    for (int64_t b = B - 1 - blockIdx.y; b >= 0; b -= gridDim.y) {
        const bool tok_ok = in_range(111, b, 1, B);
        const bool ok = c8 < C8 && tok_ok && in_range(112, c8 * 8, 8, C);
        // the token's X and F_out are requested (into L2, no registers held)
        // before its coefficients, so the two round trips overlap
        if (ok) {
            const uint16_t *x = X + b * n * C + c8 * 8;
#pragma unroll
            for (int j = 0; j < n; ++j) ptx::prefetch_l2(x + j * C);
            ptx::prefetch_l2(F_out + b * C + c8 * 8);
        }
        __syncthreads();  // previous token's coefficients are no longer read
        for (int t = threadIdx.x; t < n * n + n; t += blockDim.x)
            if (tok_ok)
                hs[t] = t < n * n ? __ldg(H_res + b * n * n + t) : __ldg(H_post + b * n + (t - n * n));
        __syncthreads();
        if (ok) {
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

// Wide n: the blocks walk the tokens with the next token's coefficients
// copied into the other half of a double buffer while this one is mixed (one
// barrier a token).
template <int n, typename FT>
__global__ void __launch_bounds__(256, 2)
post_res_apply_wide_kernel(const uint16_t *X, const FT *__restrict__ F_out,
                           const float *__restrict__ H_res, const float *__restrict__ H_post,
                           int64_t B, int64_t C, uint16_t *X_next)
{
    constexpr int kH = n * n + n;
    __shared__ float hs[2][kH];
    const int64_t C8 = C >> 3;
    const int64_t c8 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const bool active = c8 < C8;
    const int64_t step = static_cast<int64_t>(gridDim.y) * n * C;  // X elements between tokens
    ptx::pdl_wait();  // H_res and H_post come from earlier kernels
    ptx::pdl_trigger();
    // coefficients of token bb into buffer k: H_res row-major, then H_post
    auto stage = [&](bool live, int64_t bb, int k) {
        if (live && in_range(121, bb, 1, B))
            for (int t = threadIdx.x; t < kH; t += blockDim.x)
                ptx::cp_async4(&hs[k][t], t < n * n ? H_res + bb * n * n + t
                                                    : H_post + bb * n + (t - n * n));
        ptx::cp_async_commit();
    };
    // The walk goes down from the last token: pre_apply, which runs just
    // before in mhc_forward, read the last tokens last, and part of their X is
    // still in L2.
    int64_t b = B - 1 - blockIdx.y;
    stage(b >= 0, b, 0);
    ptx::cp_async_wait_all();
    __syncthreads();
    for (int k = 0; b >= 0; b -= gridDim.y, k ^= 1) {
        const int64_t bn = b - gridDim.y;  // the walk's next token
        const bool next = bn >= 0;
        const uint16_t *x = X + b * n * C + c8 * 8;
        uint4 xv[n];
        float f[8];
        const bool ok = active && in_range(122, b, 1, B) && in_range(123, c8 * 8, 8, C);
        if (ok) {
#pragma unroll
            for (int j = 0; j < n; ++j) xv[j] = ptx::ld_stream_v4(x + j * C);
            load_f8(F_out + b * C + c8 * 8, f);
        }
        // buffer k ^ 1 was last read for the walk's previous token, before the
        // barrier that ended the previous step
        stage(next, bn, k ^ 1);
        if (ok && next && in_range(124, bn, 1, B)) {
#pragma unroll
            for (int j = 0; j < n; ++j) ptx::prefetch_l2(x - step + j * C);
            ptx::prefetch_l2(F_out + bn * C + c8 * 8);
        }
        if (ok) {
            uint16_t *y = X_next + b * n * C + c8 * 8;
#pragma unroll
            for (int i = 0; i < n; ++i) ptx::st_stream_v4(y + i * C, post_mix8<n>(hs[k], i, xv, f));
        }
        ptx::cp_async_wait_all();
        __syncthreads();
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

// The wide kernels' grid: a whole number of waves of resident blocks (blocks
// per SM from the occupancy calculator, kept per kernel and block size; SMs
// of the current device), the number that gives each block's walk about
// `walk` tokens, kept within [lo, hi] waves.  A partial last wave leaves SMs
// idle at the end (measured at n = 8, B = 2048: 2.24 waves 10 % slower than 2).
template <typename K>
cudaError_t wide_grid(K kernel, int64_t B, int64_t C8, int threads, int walk, int lo, int hi,
                      std::atomic<int> *cache, dim3 &grid)
{
    grid = apply_grid(B, C8, threads);
    int per_sm = cache->load(std::memory_order_relaxed);
    if (per_sm == 0) {
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) per_sm = 1;
        cache->store(per_sm, std::memory_order_relaxed);
    }
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t wave_rows = (static_cast<int64_t>(sms) * per_sm + grid.x - 1) / grid.x;
    int64_t waves = (B + walk * wave_rows / 2) / (walk * wave_rows);  // rounded to nearest
    if (waves < lo) waves = lo;
    if (waves > hi) waves = hi;
    const int64_t rows = waves * wave_rows;
    if (rows < grid.y) grid.y = static_cast<unsigned>(rows < 1 ? 1 : rows);
    return cudaSuccess;
}

// index of a block size among the ones block_threads returns
int threads_slot(int threads) { return threads == 256 ? 0 : threads == 128 ? 1 : threads == 64 ? 2 : 3; }

template <typename FT>
cudaError_t launch_post_res(const uint16_t *X, const FT *F_out, const float *H_res,
                            const float *H_post, int64_t B, int n, int64_t C, uint16_t *X_next,
                            cudaStream_t stream)
{
    const int64_t C8 = C / 8;
    const int threads = block_threads(C8);
    const dim3 grid = apply_grid(B, C8, threads);
    static std::atomic<int> per_sm[4][4];  // [n - 5][block size slot]
    switch (n) {
#define MHC_CASE(k)                                                                            \
    case k:                                                                                    \
        return launch_pdl(post_res_apply_kernel<k, FT>, grid, dim3(threads), 0, stream, X,     \
                          F_out, H_res, H_post, B, C, X_next);
        MHC_CASE(1) MHC_CASE(2) MHC_CASE(3) MHC_CASE(4)
#undef MHC_CASE
#define MHC_CASE(k)                                                                            \
    case k: {                                                                                  \
        dim3 g;                                                                                \
        const cudaError_t e = wide_grid(post_res_apply_wide_kernel<k, FT>, B, C8, threads, 6, 2, 16, \
                                        &per_sm[k - 5][threads_slot(threads)], g);             \
        if (e != cudaSuccess) return e;                                                        \
        return launch_pdl(post_res_apply_wide_kernel<k, FT>, g, dim3(threads), 0, stream, X,   \
                          F_out, H_res, H_post, B, C, X_next);                                 \
    }
        MHC_CASE(5) MHC_CASE(6) MHC_CASE(7) MHC_CASE(8)
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
    static std::atomic<int> per_sm[4][4];  // [n - 5][block size slot]
    switch (n) {
#define MHC_CASE(k) \
    case k: return launch_pdl(pre_apply_kernel<k>, grid, dim3(threads), 0, stream, X, H_pre, B, C, F_pre);
        MHC_CASE(1) MHC_CASE(2) MHC_CASE(3) MHC_CASE(4)
#undef MHC_CASE
#define MHC_CASE(k)                                                                            \
    case k: {                                                                                  \
        dim3 g;                                                                                \
        const cudaError_t e = wide_grid(pre_apply_wide_kernel<k>, B, C8, threads, 1, 32, 32,       \
                                        &per_sm[k - 5][threads_slot(threads)], g);             \
        if (e != cudaSuccess) return e;                                                        \
        return launch_pdl(pre_apply_wide_kernel<k>, g, dim3(threads), 0, stream, X, H_pre, B,  \
                          C, F_pre);                                                           \
    }
        MHC_CASE(5) MHC_CASE(6) MHC_CASE(7) MHC_CASE(8)
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
