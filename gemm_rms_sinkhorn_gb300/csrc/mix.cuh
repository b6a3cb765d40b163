// Per-token arithmetic shared by the standalone kernels and the fused one
// (page "mHC 算法分析 & cutile 高效实现", §2.3–§2.5):
//   token_coeffs  all of one token's coefficients in one thread (H_pre,
//                 H_post and the Sinkhorn–Knopp block);
//   pre_mix8      F_pre for 8 channels of one token from its n streams;
//   post_mix8     X_next for 8 channels of one token from its n streams.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace mhc {

// 1/s for the Sinkhorn normalisations and the sigmoids: the hardware's
// approximate reciprocal, within one ulp of the exact 1/s over the normal
// range (the PTX ISA's bound for rcp.approx; a GPU test checks it), flushing
// subnormal inputs and results to zero.  The row and column sums are always
// normal: every row holds its maximum, exp(0) = 1, before the first step.
// One instruction without a branch, so the n reciprocals of a row or column
// step overlap, where a correctly rounded division's slow-path branch
// serialises them.
__device__ __forceinline__ float recip_approx(float s)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(s));
    return y;
}

// σ(x) = 1/(1 + e^{−x}) with the reciprocal above.  For x below about −88,
// e^{−x} overflows; the clamp keeps the reciprocal finite, and its value
// (below the smallest normal float) flushes to the exact limit 0.
__device__ __forceinline__ float sigmoid(float x)
{
    return recip_approx(fminf(1.0f + expf(-x), 3.0e38f));
}

// §2.3 + §2.4 for one pre entry: H_pre = σ(α_pre·y·(1/r) + b).  inv_r is the
// token's 1/r; every caller forms it as 1.0f / r, so all get the same bits.
__device__ __forceinline__ float pre_coeff(float y, float inv_r, float a_pre, float b)
{
    return sigmoid(a_pre * y * inv_r + b);
}

// Σ v[0..k) as a balanced tree (depth ⌈log2 k⌉, which shortens the
// Sinkhorn step's dependency chain).
template <int k>
__device__ __forceinline__ float tree_sum(const float *v)
{
    if constexpr (k == 1) {
        return v[0];
    } else {
        constexpr int h = k / 2;
        return tree_sum<h>(v) + tree_sum<k - h>(v + h);
    }
}

// All coefficients of one token in one thread.  y: the token's N = n²+2n raw
// coefficients; rb: its r.
//   §2.3  H̃ = α_seg·y/r + b, with y/r formed as y·(1/r): one division a token
//         (a division's slow-path branch keeps n²+2n of them from overlapping)
//   §2.4  hp = σ(H̃_pre), hq = 2σ(H̃_post); m = Sinkhorn–Knopp(exp H̃_res)
// The n×n block stays in registers, so row and column sums are thread-local
// (pairwise tree sums).  Each normalisation multiplies by one reciprocal of
// the sum.  Rows are shifted by their maximum before exp when iters > 0:
// exp(h − mx)/Σ exp(h − mx) = exp(h)/Σ exp(h), so every iterate from the first
// row step on is unchanged in exact arithmetic while exp cannot overflow;
// iters = 0 returns the raw exp(H̃_res).
template <int n>
__device__ __forceinline__ void token_coeffs(const float *y, float rb, const float *bias,
                                             float a_pre, float a_post, float a_res, int iters,
                                             float (&hp)[n], float (&hq)[n], float (&m)[n][n])
{
    const float inv_r = 1.0f / rb;
#pragma unroll
    for (int i = 0; i < n; ++i) {
        hp[i] = pre_coeff(y[i], inv_r, a_pre, bias[i]);
        hq[i] = 2.0f * sigmoid(a_post * y[n + i] * inv_r + bias[n + i]);
    }
#pragma unroll
    for (int i = 0; i < n; ++i)
#pragma unroll
        for (int j = 0; j < n; ++j)
            m[i][j] = a_res * y[2 * n + i * n + j] * inv_r + bias[2 * n + i * n + j];
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
    if constexpr (n <= 4) {
        // rows, then columns, scaled in place
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int i = 0; i < n; ++i) {
                const float inv = recip_approx(tree_sum<n>(m[i]));
#pragma unroll
                for (int j = 0; j < n; ++j) m[i][j] *= inv;
            }
#pragma unroll
            for (int j = 0; j < n; ++j) {
                float col[n];
#pragma unroll
                for (int i = 0; i < n; ++i) col[i] = m[i][j];
                const float inv = recip_approx(tree_sum<n>(col));
#pragma unroll
                for (int i = 0; i < n; ++i) m[i][j] *= inv;
            }
        }
    } else {
        // The same iteration kept as diagonal scalings of the fixed A = m:
        // after each step the iterate is diag(u)·A·diag(v), the row step sets
        // u_i = 1/Σ_j A_ij·v_j and the column step v_j = 1/Σ_i u_i·A_ij.  It does
        // no n² rescaling per step, which measured 1.3–2.5× faster per
        // iteration on GB300 for n = 5..8 (the in-place form is faster at n <= 4).
        if (iters > 0) {
            float u[n], v[n];
#pragma unroll
            for (int j = 0; j < n; ++j) v[j] = 1.0f;
            for (int it = 0; it < iters; ++it) {
#pragma unroll
                for (int i = 0; i < n; ++i) {
                    float p[n];
#pragma unroll
                    for (int j = 0; j < n; ++j) p[j] = m[i][j] * v[j];
                    u[i] = recip_approx(tree_sum<n>(p));
                }
#pragma unroll
                for (int j = 0; j < n; ++j) {
                    // products rounded on their own (never fused into the sum's
                    // adds), so a column sum split across lanes gives these bits
                    float p[n];
#pragma unroll
                    for (int i = 0; i < n; ++i) p[i] = __fmul_rn(u[i], m[i][j]);
                    v[j] = recip_approx(tree_sum<n>(p));
                }
            }
#pragma unroll
            for (int i = 0; i < n; ++i)
#pragma unroll
                for (int j = 0; j < n; ++j) m[i][j] = (u[i] * m[i][j]) * v[j];
        }
    }
}

// token_coeffs for one token on a pair of adjacent lanes (lane parity =
// half): half 0 takes rows [0, n/2) of H_res and those entries of H_pre and
// H_post, half 1 rows [n/2, n), and each stores its own (when `store`).  Row
// steps are local.  A column sum is the two halves' partial tree sums added,
// which is exactly how tree_sum<n> splits (tree_sum<n/2> + tree_sum<n - n/2>),
// and every other value is the same expression on the same operands, so the
// result equals token_coeffs' to the bit (the column products are rounded
// on their own in both, so no add fuses one of them in one form and not the
// other).  Every lane of the warp must call it
// (the column sums cross lanes); a lane with nothing to store passes
// store = false.  n >= 2.
template <int n>
__device__ __forceinline__ void token_coeffs_pair(const float *y, float rb, const float *bias,
                                                  float a_pre, float a_post, float a_res,
                                                  int iters, int half, bool store, int64_t t,
                                                  float *H_pre, float *H_post, float *H_res)
{
    static_assert(n >= 2, "a pair needs a row for each half");
    constexpr int h0 = n / 2, kR = n - n / 2;  // rows of half 0; rows of half 1
    const int i0 = half ? h0 : 0;
    const int cnt = half ? kR : h0;
    const float inv_r = 1.0f / rb;
    // the other half's partial of a column sum, added in tree_sum<n>'s order
    const auto col_total = [&](const float (&p)[kR]) {
        const float own = half ? tree_sum<kR>(p) : tree_sum<h0>(p);
        const float other = __shfl_xor_sync(0xffffffffu, own, 1);
        return half ? other + own : own + other;
    };
    float m[kR][n];
#pragma unroll
    for (int r = 0; r < kR; ++r) {
        const int i = r < cnt ? i0 + r : i0;  // a spare row (half 0, odd n) repeats row i0
#pragma unroll
        for (int j = 0; j < n; ++j)
            m[r][j] = a_res * y[2 * n + i * n + j] * inv_r + bias[2 * n + i * n + j];
    }
    if (iters > 0) {
#pragma unroll
        for (int r = 0; r < kR; ++r) {
            float mx = m[r][0];
#pragma unroll
            for (int j = 1; j < n; ++j) mx = fmaxf(mx, m[r][j]);
#pragma unroll
            for (int j = 0; j < n; ++j) m[r][j] = expf(m[r][j] - mx);
        }
    } else {
#pragma unroll
        for (int r = 0; r < kR; ++r)
#pragma unroll
            for (int j = 0; j < n; ++j) m[r][j] = expf(m[r][j]);
    }
    if constexpr (n <= 4) {
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int r = 0; r < kR; ++r) {
                const float inv = recip_approx(tree_sum<n>(m[r]));
#pragma unroll
                for (int j = 0; j < n; ++j) m[r][j] *= inv;
            }
#pragma unroll
            for (int j = 0; j < n; ++j) {
                float col[kR];
#pragma unroll
                for (int r = 0; r < kR; ++r) col[r] = m[r][j];
                const float inv = recip_approx(col_total(col));
#pragma unroll
                for (int r = 0; r < kR; ++r) m[r][j] *= inv;
            }
        }
    } else {
        if (iters > 0) {
            float u[kR], v[n];
#pragma unroll
            for (int j = 0; j < n; ++j) v[j] = 1.0f;
            for (int it = 0; it < iters; ++it) {
#pragma unroll
                for (int r = 0; r < kR; ++r) {
                    float p[n];
#pragma unroll
                    for (int j = 0; j < n; ++j) p[j] = m[r][j] * v[j];
                    u[r] = recip_approx(tree_sum<n>(p));
                }
#pragma unroll
                for (int j = 0; j < n; ++j) {
                    float p[kR];
#pragma unroll
                    for (int r = 0; r < kR; ++r) p[r] = __fmul_rn(u[r], m[r][j]);
                    v[j] = recip_approx(col_total(p));
                }
            }
#pragma unroll
            for (int r = 0; r < kR; ++r)
#pragma unroll
                for (int j = 0; j < n; ++j) m[r][j] = (u[r] * m[r][j]) * v[j];
        }
    }
    if (!store) return;
#pragma unroll
    for (int r = 0; r < kR; ++r) {
        if (r >= cnt) break;
        const int i = i0 + r;
        H_pre[t * n + i] = pre_coeff(y[i], inv_r, a_pre, bias[i]);
        H_post[t * n + i] = 2.0f * sigmoid(a_post * y[n + i] * inv_r + bias[n + i]);
        float *o = H_res + (t * n + i) * n;
        if constexpr (n % 4 == 0) {
#pragma unroll
            for (int j = 0; j < n; j += 4)
                *reinterpret_cast<float4 *>(o + j) =
                    make_float4(m[r][j], m[r][j + 1], m[r][j + 2], m[r][j + 3]);
        } else {
#pragma unroll
            for (int j = 0; j < n; ++j) o[j] = m[r][j];
        }
    }
}

// Stores one token's coefficients (row-major H_res), 128-bit where the
// per-token strides keep 16-byte alignment.
template <int n>
__device__ __forceinline__ void store_token_coeffs(int64_t t, const float (&hp)[n],
                                                   const float (&hq)[n], const float (&m)[n][n],
                                                   float *H_pre, float *H_post, float *H_res)
{
    if constexpr (n % 4 == 0) {
#pragma unroll
        for (int i = 0; i < n; i += 4) {
            *reinterpret_cast<float4 *>(H_pre + t * n + i) =
                make_float4(hp[i], hp[i + 1], hp[i + 2], hp[i + 3]);
            *reinterpret_cast<float4 *>(H_post + t * n + i) =
                make_float4(hq[i], hq[i + 1], hq[i + 2], hq[i + 3]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < n; ++i) {
            H_pre[t * n + i] = hp[i];
            H_post[t * n + i] = hq[i];
        }
    }
    float *o = H_res + t * n * n;
    if constexpr ((n * n) % 4 == 0) {
        // row-major flat index k = i·n + j, four at a time
#pragma unroll
        for (int k = 0; k < n * n; k += 4)
            *reinterpret_cast<float4 *>(o + k) =
                make_float4(m[k / n][k % n], m[(k + 1) / n][(k + 1) % n],
                            m[(k + 2) / n][(k + 2) % n], m[(k + 3) / n][(k + 3) % n]);
    } else {
#pragma unroll
        for (int i = 0; i < n; ++i)
#pragma unroll
            for (int j = 0; j < n; ++j) o[i * n + j] = m[i][j];
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

// The channel pairs (2p, 2p+1) of 8 bf16 channels, each pair as two fp32 lanes.
__device__ __forceinline__ void unpack8_pairs(const uint4 &v, uint64_t (&t)[4])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int p = 0; p < 4; ++p) t[p] = f2_pack(bf16_lo(w[p]), bf16_hi(w[p]));
}

__device__ __forceinline__ uint4 pack8_pairs(const uint64_t (&acc)[4])
{
    float f[8];
#pragma unroll
    for (int p = 0; p < 4; ++p) f2_unpack(acc[p], f[2 * p], f[2 * p + 1]);
    return pack8(f);
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

// §2.5 (2): row i of X_next for 8 channels, Σ_j H_res[i][j]·X[j] + H_post[i]·F_out,
// fp32, rounded to bf16 (RNE).  hs: H_res row-major (n·n) followed by H_post (n).
// Each channel's chain is taken in the same order either way.  Wide n runs
// packed multiply-adds on channel pairs (n² + n FMAs a channel make the
// instruction count matter there); up to n = 4 the kernel is bound by memory
// and the register pairs would spill under its 64-register cap (measured at
// n = 8: 2-2.5 % faster X_next, at C = 4096 and 7168).
template <int n>
__device__ __forceinline__ uint4 post_mix8(const float *hs, int i, const uint4 (&xv)[n],
                                           const float (&f)[8])
{
    if constexpr (n <= 4) {
        float acc[8], t[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
        for (int j = 0; j < n; ++j) {
            const float hij = hs[i * n + j];
            unpack8(xv[j], t);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(hij, t[e], acc[e]);
        }
        const float hq = hs[n * n + i];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(hq, f[e], acc[e]);
        return pack8(acc);
    } else {
        uint64_t acc[4], t[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) acc[p] = 0;  // +0, +0
#pragma unroll
        for (int j = 0; j < n; ++j) {
            const float hij = hs[i * n + j];
            const uint64_t hh = f2_pack(hij, hij);
            unpack8_pairs(xv[j], t);
#pragma unroll
            for (int p = 0; p < 4; ++p) acc[p] = f2_fma(hh, t[p], acc[p]);
        }
        const float hq = hs[n * n + i];
        const uint64_t qq = f2_pack(hq, hq);
#pragma unroll
        for (int p = 0; p < 4; ++p) acc[p] = f2_fma(qq, f2_pack(f[2 * p], f[2 * p + 1]), acc[p]);
        return pack8_pairs(acc);
    }
}

}  // namespace mhc
