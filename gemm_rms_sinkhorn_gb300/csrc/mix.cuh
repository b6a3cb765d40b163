// Per-token arithmetic shared by the standalone kernels and the fused one
// (page "mHC 算法分析 & cutile 高效实现", §2.3–§2.5):
//   coeff_lane  one lane's share of a token's coefficients: entries i of H_pre
//               and H_post and row i of the Sinkhorn–Knopp block;
//   pre_mix8    F_pre for 8 channels of one token from its n streams.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace mhc {

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

// §2.3 + §2.4 for one pre entry: H_pre = σ(α_pre·y/r + b).  The expression
// leaves the compiler nothing to contract, so every caller gets the same bits.
__device__ __forceinline__ float pre_coeff(float y, float rb, float a_pre, float b)
{
    return 1.0f / (1.0f + expf(-(a_pre * y / rb + b)));
}

// Lane i of the n-lane group of one token (lanes base..base+n-1 of the warp,
// all in `mask`).  y: the token's N = n²+2n raw coefficients; rb: its r.
//   §2.3  H̃ = α_seg·y/r + b
//   §2.4  hp = σ(H̃_pre[i]), hq = 2σ(H̃_post[i]); m = row i of Sinkhorn(exp H̃_res)
// The n×n block is row-distributed over the lanes; each normalisation
// multiplies by one correctly rounded reciprocal of the sum.  Rows are shifted
// by their maximum before exp when iters > 0 (exact after the first row
// normalisation); iters = 0 returns the raw exp(H̃_res).
template <int n>
__device__ __forceinline__ void coeff_lane(const float *y, float rb, const float *bias, float a_pre,
                                           float a_post, float a_res, int iters, int i, int base,
                                           unsigned mask, float &hp, float &hq, float (&m)[n])
{
    hp = pre_coeff(y[i], rb, a_pre, bias[i]);
    hq = 2.0f / (1.0f + expf(-(a_post * y[n + i] / rb + bias[n + i])));
#pragma unroll
    for (int j = 0; j < n; ++j) m[j] = a_res * y[2 * n + i * n + j] / rb + bias[2 * n + i * n + j];
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
}

__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8])
{
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8])
{
    return make_uint4(pack_bf16_rn(f[0], f[1]), pack_bf16_rn(f[2], f[3]),
                      pack_bf16_rn(f[4], f[5]), pack_bf16_rn(f[6], f[7]));
}

// §2.5 (1): 8 channels of F_pre = Σ_i h[i]·X[i], fp32, rounded to bf16 (RNE).
template <int n>
__device__ __forceinline__ uint4 pre_mix8(const float (&h)[n], const uint4 (&xv)[n])
{
    float acc[8], t[8];
    unpack8(xv[0], t);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = h[0] * t[e];
#pragma unroll
    for (int i = 1; i < n; ++i) {
        unpack8(xv[i], t);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(h[i], t[e], acc[e]);
    }
    return pack8(acc);
}

}  // namespace mhc
