// Steps 1 to 4a of the mHC forward in one launch for small batches (decode):
// the projection GEMM with the RMS (§2.1, §2.2), the coefficients and the
// Sinkhorn–Knopp projection (§2.3, §2.4), and F_pre (§2.5 (1)), page "mHC 算法
// 分析 & cutile 高效实现".  With a few tokens the forward is a chain of
// latencies, not of bytes (§3.2 counts the launches, §5.1 the idle SMs), so
// this kernel replaces the chain's launches by one and spreads the GEMM over every SM.
//
//   phase 1  the stream-K X·φ + Σx² pipeline of gemm_pipeline.cuh over all SMs;
//            every CTA parks its partial sums (one slot per CTA and token tile);
//   barrier  a grid-wide arrival count (the launch is cooperative, so every CTA
//            is resident), bounded like every other wait;
//   phase 2  CTA c owns the items [c·T/G, (c+1)·T/G) of the T = B·C/8 pieces
//            of 8 channels, token-major.  For each token its items touch it
//            sums the partials over the tile's contributors in a fixed order
//            (segments of 32 contributors in index order, then the segments in
//            index order), so every CTA that needs a token gets the same bits,
//            then runs token_coeffs (one thread per token); the CTA owning the
//            token's first item writes Y, r, H_pre, H_post and H_res;
//   phase 3  F_pre of its items from X, which phase 1 has just streamed
//            through L2, by nine warps while the tenth runs the Sinkhorn
//            iteration (F_pre needs only H_pre, a sigmoid of the totals);
//   phase 4  (when X_next is given) X_next (§2.5 (2)) of the same items, by
//            all ten warps, once the Sinkhorn iteration has given H_res.
//            mhc_forward takes F_out as an input, so it is there from the
//            start (in a layer, where F_out = F(F_pre), the step entry points
//            run S4b after F).  Each item is read and written by one thread
//            only, so X_next may be X.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>
#include <random>
#include <type_traits>

#include "check.cuh"
#include "gemm_pipeline.cuh"
#include "mhc_internal.h"
#include "mix.cuh"
#include "ptx.cuh"

namespace mhc {
namespace {

using pipe::kBK;
using pipe::kBM;
using pipe::Sched;
using pipe::Segment;
using pipe::SegIter;

constexpr int kThreads = 320;  // 10 warps: TMA, MMA, 4 × square-sum, 4 × epilogue
constexpr int kRingBudget = 160 * 1024;
constexpr int kMaxTokens = 4096;  // largest batch this path takes
constexpr int kSegLen = 32;       // contributors per first-level segment of the sum
constexpr int kRedFloats = 16384; // first-level segment sums of one token batch
constexpr int kTokBatch = 32;     // tokens whose coefficients are formed together

__device__ int g_decode_status;

constexpr int npad_for(int n) { return (n * n + 2 * n + 15) / 16 * 16; }

// kSplit: the weight operand is the fp32-weight form (bf16 pairs, 2N rows;
// see launch_gemm_rms_split) and the epilogue adds each pair of columns.
template <int n, bool kSplit>
struct DCfg {
    static constexpr int N = n * n + 2 * n;
    static constexpr int V = N + 1;  // a partial row: N sums of products, then Σx²
    static constexpr int kH = n * n + n;  // a token's H_res (row-major), then H_post
    using FT = std::conditional_t<kSplit, float, uint16_t>;  // the element type of F_out
    static constexpr int NPAD = kSplit ? (2 * N + 15) / 16 * 16 : npad_for(n);
    using C = pipe::Cfg<NPAD, kRingBudget>;
    static constexpr int kBiasBytes = (N * 4 + 15) / 16 * 16;  // b, staged for phase 2
    static constexpr int kSmemBytes =
        1024 + C::kRingBytes + pipe::kSsBytes + pipe::kBarrierBytes + kBiasBytes;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
    // phase 2 scratch reuses the stage ring
    static_assert((kRedFloats + kTokBatch * V + kTokBatch * n + kTokBatch * 4 + kTokBatch * kH) *
                      4 <= C::kRingBytes, "scratch");
};

constexpr int kMaxTiles = kMaxTokens / kBM;

// The contributors (CTAs) first[m]..last[m] of each token tile, from the host.
struct TileCtas {
    int first[kMaxTiles], last[kMaxTiles];
};

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

// The grid barrier's two words (arrivals, then departures) hold a launch's
// 48-bit epoch above a 16-bit count.  CTA 0 writes (epoch, 0) to both as it
// starts, once the previous kernel has finished, so the words need no clearing
// beforehand.  An arrival is one atomic add; one that lands before CTA 0's
// write (the old value carries another tag) is wiped out by that write and is
// made again.  The last CTA to leave, and every CTA whose wait runs out, set
// both words to 0, so no later launch meets this launch's tag, not even a
// replay of the same CUDA graph, which reuses the epoch.
constexpr int kCountBits = 16;
constexpr unsigned long long kCountMask = (1ull << kCountBits) - 1;

__device__ __forceinline__ bool tagged(unsigned long long v, unsigned long long epoch)
{
    return (v >> kCountBits) == epoch;
}

// Adds this CTA's arrival to *w for this epoch; false when the word did not
// carry the epoch before the limit ran out (counted from t0).
__device__ bool arrive(unsigned long long *w, unsigned long long epoch, uint64_t t0,
                       uint64_t limit_ns)
{
    for (;;) {
        if (tagged(atomicAdd(w, 1ull), epoch)) return true;
        for (uint32_t polls = 0; !tagged(ptx::ld_acquire_gpu_u64(w), epoch); ++polls) {
            if ((polls & 31) == 31 && ptx::globaltimer_ns() - t0 > limit_ns) return false;
            __nanosleep(64);
        }
        if (ptx::globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// Bounded spin until *w counts at least `target` for this epoch; false when
// the limit ran out (counted from t0).
__device__ bool wait_arrivals(const unsigned long long *w, unsigned long long epoch,
                              uint32_t target, uint64_t t0, uint64_t limit_ns)
{
    for (uint32_t polls = 0;; ++polls) {
        const unsigned long long v = ptx::ld_acquire_gpu_u64(w);
        if (tagged(v, epoch) && (v & kCountMask) >= target) return true;
        if ((polls & 31) == 31 && ptx::globaltimer_ns() - t0 > limit_ns) return false;
        __nanosleep(32);
    }
}

template <int n, bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
decode_pre_kernel(const __grid_constant__ CUtensorMap tm_x,
                  const __grid_constant__ CUtensorMap tm_w, const uint16_t *X,
                  int64_t B, int64_t C, Sched sch, const __grid_constant__ TileCtas tc,
                  int seg_max, float a_pre, float a_post, float a_res,
                  const float *__restrict__ bias, int iters, float *__restrict__ Y,
                  float *__restrict__ r, float *__restrict__ H_pre, float *__restrict__ H_post,
                  float *__restrict__ H_res, uint16_t *__restrict__ F_pre,
                  const typename DCfg<n, kSplit>::FT *__restrict__ F_out, uint16_t *X_next,
                  float *__restrict__ partials, unsigned long long *grid_bar,
                  unsigned long long epoch, uint32_t bar_target, uint64_t wait_limit_ns)
{
    using D = DCfg<n, kSplit>;
    using Cf = typename D::C;
    constexpr int N = D::N, V = D::V, NPAD = D::NPAD, kH = D::kH;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    pipe::Pipe p;
    float *bias_s = reinterpret_cast<float *>(
        pipe::carve<NPAD, kRingBudget>(p, smem, &g_decode_status, wait_limit_ns));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const int64_t K = n * C;
    // partial rows of the workspace: one slot of kBM rows per CTA and tile
    const int64_t part_rows = (static_cast<int64_t>(sch.grid) + sch.m_tiles) * kBM;
    // this CTA's items for phases 2-3 (64-bit divisions: done here, before the
    // previous kernel has finished, not on the path after the grid barrier)
    const int64_t C8 = C >> 3;
    const int64_t T = B * C8;
    const int64_t lo = T * cta / sch.grid, hi = T * (cta + 1) / sch.grid;
    const int64_t t_first = lo / C8, t_last = (hi - 1) / C8;

    if (threadIdx.x == 0) {
        pipe::init_barriers(p);
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tm_x);
        ptx::prefetch_tensormap(&tm_w);
    }
    if (warp == 1) ptx::tmem_alloc<Cf::kTmemCols>(p.tmem_holder);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    p.tmem_base = *p.tmem_holder;
    ptx::pdl_wait();
    if (cta == 0 && threadIdx.x == 0) {  // this launch's tag on the grid barrier's words
        atomicExch(grid_bar + 1, epoch << kCountBits);
        __threadfence();
        atomicExch(grid_bar, epoch << kCountBits);
    }
    // b for phase 2, fetched now so its latency hides behind phase 1
    for (int k = threadIdx.x; k < N; k += kThreads) bias_s[k] = __ldg(bias + k);

    // ------------------------------------------------------------ phase 1
    const SegIter segs{sch.lo(cta), sch.lo(cta + 1), sch.kbt};
    if (warp == 0) {
        if (lane == 0)  // X is read again in phase 3 and by the X_next kernel: keep it in L2
            pipe::producer<NPAD>(p, segs, &tm_x, &tm_w, ptx::policy_evict_normal(), -1);
    } else if (warp == 1) {
        if (lane == 0) pipe::mma_issuer<NPAD>(p, segs);
    } else if (warp < 6) {
        pipe::square_sum<NPAD>(p, segs, (warp - 2) * 32 + lane, lane);
    } else {
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        int seg = 0;
        SegIter it = segs;
        Segment sg;
        while (it.next(sg)) {
            const int64_t grow = static_cast<int64_t>(sg.m) * kBM + row;
            const int64_t prow = static_cast<int64_t>(cta + sg.m) * kBM + row;
            float *mine = partials + prow * V;
            // a row past B stores nothing; one inside must have its slot
            const bool keep = grow < B && in_range(601, prow, 1, part_rows);
            float ss;
            if constexpr (kSplit) {
                const bool ok = pipe::take_accumulator_chunked<NPAD>(
                    p, seg, q, lane, ss, [&](int c, const float (&v)[32]) {
                        if (!keep) return;
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            if (c * 16 + e < N) mine[c * 16 + e] = v[2 * e] + v[2 * e + 1];
                    });
                if (!ok) break;
            } else {
                float v[NPAD];
                if (!pipe::take_accumulator<NPAD>(p, seg, q, lane, v, ss)) break;
                if (keep) {
#pragma unroll
                    for (int j = 0; j < NPAD; ++j)
                        if (j < N) mine[j] = v[j];
                }
            }
            ++seg;
            if (keep) mine[N] = ss;
        }
    }
    // lane 0 of the TMA and MMA warps ran alone: reconverge every warp before
    // the CTA barrier, which needs whole warps
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc<Cf::kTmemCols>(p.tmem_base);
    }

    // ------------------------------------------------------ grid barrier
    // The CTA barrier above orders every thread's partial stores before thread
    // 0's fence, which is cumulative: they are visible before its arrival.
    if (threadIdx.x == 0) {
        __threadfence();
        unsigned long long *departed = grid_bar + 1;
        // A CTA whose phase 1 gave up still arrives and leaves like the
        // others (they are all resident, so its wait is short) and returns
        // below; only a wait that runs out clears the words early.
        const uint64_t t0 = ptx::globaltimer_ns();
        if (!arrive(grid_bar, epoch, t0, wait_limit_ns) ||
            !wait_arrivals(grid_bar, epoch, bar_target, t0, wait_limit_ns)) {
            atomicExch(grid_bar, 0ull);  // leave the words clear for the next launch
            atomicExch(departed, 0ull);
            pipe::raise_timeout(p);
        } else {
            const unsigned long long left = atomicAdd(departed, 1ull);
            if (tagged(left, epoch) && (left & kCountMask) + 1 == gridDim.x) {
                // every CTA has seen the barrier complete: clear it for the next launch
                atomicExch(grid_bar, 0ull);
                atomicExch(departed, 0ull);
            }
        }
    }
    __syncwarp();  // warp 0 whole again before the CTA barrier
    __syncthreads();
    if (*p.abort) return;
    // the X_next kernel may start launching; it waits for this grid to finish
    ptx::pdl_trigger();

    // -------------------------------------------------- phases 2 and 3
    if (lo >= hi) return;
    float *red = reinterpret_cast<float *>(p.stages);  // [seg_max][tokens · V]
    float *yv = red + kRedFloats;                      // [tokens][V]: Y row, then r
    float *hps = yv + kTokBatch * V;                   // [tokens][n]: H_pre
    int *tinfo = reinterpret_cast<int *>(hps + kTokBatch * n);  // [tokens]: first, last, m, row
    float *hres = reinterpret_cast<float *>(tinfo + kTokBatch * 4);  // [tokens][kH]: H_res, H_post
    int nb = kRedFloats / (V * seg_max);
    if (nb > kTokBatch) nb = kTokBatch;
    for (int64_t t0 = t_first; t0 <= t_last; t0 += nb) {
        const int cnt = static_cast<int>(t_last - t0 + 1 < nb ? t_last - t0 + 1 : nb);
        if (threadIdx.x < cnt) {
            const int64_t t = t0 + threadIdx.x;
            int m = static_cast<int>(t / kBM);
            if (!in_range(602, m, 1, sch.m_tiles < kMaxTiles ? sch.m_tiles : kMaxTiles)) m = 0;
            int *ti = tinfo + threadIdx.x * 4;
            ti[0] = tc.first[m];
            ti[1] = tc.last[m];
            ti[2] = m;
            ti[3] = static_cast<int>(t - static_cast<int64_t>(m) * kBM);
        }
        __syncthreads();
        // first level: segment s of value v of token j sums contributors
        // first + s·kSegLen ... (at most kSegLen of them) in index order.  The
        // value index varies fastest across threads, so a warp's loads of one
        // contributor are one contiguous partial row.
        const int Q = cnt * V;
        const int pairs = Q * seg_max;
        for (int pi = threadIdx.x; pi < pairs; pi += kThreads) {
            const int s = pi / Q, qv = pi - s * Q;
            const int j = qv / V, v = qv - j * V;
            const int *ti = tinfo + j * 4;
            const int last = ti[1], m = ti[2], row = ti[3];
            const int c0 = ti[0] + s * kSegLen;
            float acc = 0.f;
            if (c0 <= last && in_range(603, (static_cast<int64_t>(last + m) * kBM + row), 1,
                                       part_rows)) {
                float vals[kSegLen];
#pragma unroll
                for (int u = 0; u < kSegLen; ++u)
                    vals[u] = c0 + u <= last
                                  ? __ldcg(partials + (static_cast<int64_t>(c0 + u + m) * kBM + row) * V + v)
                                  : 0.f;
                acc = vals[0];
#pragma unroll
                for (int u = 1; u < kSegLen; ++u) acc += vals[u];
            }
            if (in_range(604, pi, 1, kRedFloats)) red[pi] = acc;
        }
        __syncthreads();
        // second level: the segments in index order; Y and r of owned tokens
        for (int qv = threadIdx.x; qv < cnt * V; qv += kThreads) {
            const int j = qv / V, v = qv - j * V;
            const int64_t t = t0 + j;
            const int segs_t = (tinfo[j * 4 + 1] - tinfo[j * 4] + kSegLen) / kSegLen;
            float tot = red[qv];
            for (int s = 1; s < segs_t; ++s) tot += red[s * cnt * V + qv];
            // this CTA holds the token's first item
            const bool owner = t * C8 >= lo && in_range(605, t, 1, B);
            if (v < N) {
                yv[qv] = tot;
                if (owner) Y[t * N + v] = tot;
            } else {
                const float rr = sqrtf(tot / static_cast<float>(K));
                yv[qv] = rr;
                if (owner) r[t] = rr;
            }
        }
        __syncthreads();
        // H_pre first (σ of the pre entries only), so that F_pre can be formed
        // while the Sinkhorn iteration runs; token_coeffs forms the same bits
        if (threadIdx.x < cnt * n) {
            const int j = threadIdx.x / n, i = threadIdx.x - j * n;
            hps[threadIdx.x] = pre_coeff(yv[j * V + i], 1.0f / yv[j * V + N], a_pre, bias_s[i]);
        }
        __syncthreads();
        if (warp == kThreads / 32 - 1) {
            // coefficients, one lane per token (cnt <= kTokBatch = 32)
            if (lane < cnt) {
                const int64_t t = t0 + lane;
                float hp[n], hq[n], mres[n][n];
                token_coeffs<n>(yv + lane * V, yv[lane * V + N], bias_s, a_pre, a_post, a_res,
                                iters, hp, hq, mres);
                if (t * C8 >= lo && in_range(606, t, 1, B))
                    store_token_coeffs<n>(t, hp, hq, mres, H_pre, H_post, H_res);
                // for phase 4
                float *hr = hres + lane * kH;
#pragma unroll
                for (int i = 0; i < n; ++i) {
#pragma unroll
                    for (int jj = 0; jj < n; ++jj) hr[i * n + jj] = mres[i][jj];
                    hr[n * n + i] = hq[i];
                }
            }
        } else {
            // F_pre of this CTA's items of these tokens, token by token, kU
            // items a thread at a time so that their loads are in flight together
            constexpr int kMixThreads = kThreads - 32;
            constexpr int kU = n <= 4 ? 4 : (n <= 6 ? 2 : 1);
            for (int j = 0; j < cnt; ++j) {
                const int64_t t = t0 + j;
                const int64_t a = (t * C8 > lo ? t * C8 : lo) - t * C8;
                const int64_t b = ((t + 1) * C8 < hi ? (t + 1) * C8 : hi) - t * C8;
                float h[n];
#pragma unroll
                for (int i = 0; i < n; ++i) h[i] = hps[j * n + i];
                const uint16_t *xt = X + t * n * C;
                uint16_t *ft = F_pre + t * C;
                if (!in_range(607, t, 1, B) || !in_range(608, a * 8, (b > a ? b - a : 0) * 8, C)) continue;
                for (int64_t c0 = a + threadIdx.x; c0 < b; c0 += kMixThreads * kU) {
                    uint4 xv[kU][n];
#pragma unroll
                    for (int u = 0; u < kU; ++u) {
                        const int64_t c8 = c0 + u * kMixThreads;
                        if (c8 < b) {
#pragma unroll
                            for (int i = 0; i < n; ++i)  // plain loads: X_next may be X
                                xv[u][i] = *reinterpret_cast<const uint4 *>(xt + i * C + c8 * 8);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < kU; ++u) {
                        const int64_t c8 = c0 + u * kMixThreads;
                        if (c8 < b) ptx::st_stream_v4(ft + c8 * 8, pre_mix8<n>(h, xv[u]));
                    }
                }
            }
        }
        if (X_next != nullptr) {
            __syncthreads();  // H_res and H_post of the batch are in shared memory
            // phase 4: X_next of this CTA's items of these tokens, by all ten
            // warps, kV items a thread at a time so that their loads are in
            // flight together; every item's loads come before its stores, in
            // the same thread
            constexpr int kV = n <= 3 ? 2 : 1;
            for (int j = 0; j < cnt; ++j) {
                const int64_t t = t0 + j;
                const int64_t a = (t * C8 > lo ? t * C8 : lo) - t * C8;
                const int64_t b = ((t + 1) * C8 < hi ? (t + 1) * C8 : hi) - t * C8;
                if (!in_range(609, t, 1, B) || !in_range(610, a * 8, (b > a ? b - a : 0) * 8, C))
                    continue;
                const float *hr = hres + j * kH;
                const uint16_t *xt = X + t * n * C;
                const typename D::FT *fo = F_out + t * C;
                uint16_t *yt = X_next + t * n * C;
                for (int64_t c0 = a + threadIdx.x; c0 < b; c0 += kThreads * kV) {
                    uint4 xv[kV][n];
                    float f[kV][8];
#pragma unroll
                    for (int u = 0; u < kV; ++u) {
                        const int64_t c8 = c0 + u * kThreads;
                        if (c8 < b) {
#pragma unroll
                            for (int i = 0; i < n; ++i) xv[u][i] = ptx::ld_stream_v4(xt + i * C + c8 * 8);
                            load_f8(fo + c8 * 8, f[u]);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < kV; ++u) {
                        const int64_t c8 = c0 + u * kThreads;
                        if (c8 < b) {
#pragma unroll
                            for (int i = 0; i < n; ++i)
                                ptx::st_stream_v4(yt + i * C + c8 * 8, post_mix8<n>(hr, i, xv[u], f[u]));
                        }
                    }
                }
            }
        }
        __syncthreads();  // the scratch is reused by the next token batch
    }
}

Sched decode_sched(int64_t B, int n, int64_t C, int num_sms)
{
    Sched s;
    s.m_tiles = static_cast<int>((B + kBM - 1) / kBM);
    s.kbt = static_cast<int>((n * C + kBK - 1) / kBK);
    s.total = static_cast<int64_t>(s.m_tiles) * s.kbt;
    s.grid = static_cast<int>(s.total < num_sms ? s.total : num_sms);
    return s;
}

TileCtas tile_ctas(const Sched &s)
{
    TileCtas tc{};
    for (int m = 0; m < s.m_tiles; ++m) {
        tc.first[m] = s.owner(static_cast<int64_t>(m) * s.kbt);
        tc.last[m] = s.owner(static_cast<int64_t>(m + 1) * s.kbt - 1);
    }
    return tc;
}

// Largest number of kSegLen-contributor segments of any tile.
int decode_seg_max(const Sched &s, const TileCtas &tc)
{
    int mx = 1;
    for (int m = 0; m < s.m_tiles; ++m) {
        const int segs = (tc.last[m] - tc.first[m] + kSegLen) / kSegLen;
        if (segs > mx) mx = segs;
    }
    return mx;
}

constexpr size_t kBarBytes = 256;

// A fresh 48-bit epoch per launch (never 0), from a process-wide counter that
// starts at a random value, so a stale word from another process or an
// earlier use of the memory matches it only by a 2^-48 chance.
unsigned long long next_epoch()
{
    static std::atomic<unsigned long long> counter{[] {
        std::random_device rd;
        return (static_cast<unsigned long long>(rd()) << 32) ^ rd();
    }()};
    constexpr unsigned long long kMask = (1ull << (64 - kCountBits)) - 1;
    for (;;) {
        const unsigned long long e = counter.fetch_add(1, std::memory_order_relaxed) & kMask;
        if (e != 0) return e;
    }
}

template <int n, bool kSplit>
cudaError_t launch_n(const CUtensorMap &tx, const CUtensorMap &tw, const uint16_t *X, int64_t B,
                     int64_t C, const Sched &s, const TileCtas &tc, int seg_max, float a_pre,
                     float a_post,
                     float a_res, const float *bias, int iters, float *Y, float *r, float *H_pre,
                     float *H_post, float *H_res, uint16_t *F_pre, const void *F_out,
                     uint16_t *X_next, float *partials, unsigned long long *bar,
                     unsigned long long epoch, uint32_t bar_target, uint64_t limit, int device,
                     cudaStream_t stream)
{
    using D = DCfg<n, kSplit>;
    static uint64_t configured = 0;  // one bit per device
    static std::mutex mu;
    if (device < 64 && !((configured >> device) & 1)) {
        std::lock_guard<std::mutex> lock(mu);
        cudaError_t e = cudaFuncSetAttribute(decode_pre_kernel<n, kSplit>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             D::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured |= 1ull << device;
    }
    return launch_coop_pdl(decode_pre_kernel<n, kSplit>, dim3(s.grid), dim3(kThreads), D::kSmemBytes,
                           stream, tx, tw, X, B, C, s, tc, seg_max, a_pre, a_post, a_res, bias,
                           iters, Y, r, H_pre, H_post, H_res, F_pre,
                           static_cast<const typename D::FT *>(F_out), X_next, partials, bar,
                           epoch, bar_target, limit);
}

}  // namespace

bool decode_pre_eligible(int64_t B, int n, int64_t C)
{
    return B >= 1 && B <= kMaxTokens && n >= 1 && n <= 8 && C >= 8 && C % 8 == 0;
}

size_t decode_pre_workspace_bytes(int64_t B, int n, int64_t C, int num_sms)
{
    if (!decode_pre_eligible(B, n, C)) return 0;
    const Sched s = decode_sched(B, n, C, num_sms);
    const size_t slots = static_cast<size_t>(s.grid) + s.m_tiles;
    return kBarBytes + slots * kBM * (num_coeffs(n) + 1) * sizeof(float);
}

cudaError_t launch_decode_pre(const uint16_t *X, const uint16_t *phi_t, float a_pre, float a_post,
                              float a_res, const float *bias, int iters, int64_t B, int n,
                              int64_t C, float *Y, float *r, float *H_pre, float *H_post,
                              float *H_res, uint16_t *F_pre, const void *F_out, uint16_t *X_next,
                              void *workspace, int num_sms, cudaStream_t stream,
                              uint64_t wait_limit_ns, int barrier_extra, bool split)
{
    if (!decode_pre_eligible(B, n, C)) return cudaErrorInvalidValue;
    const int N = num_coeffs(n);
    const int64_t K = n * C;
    const Sched s = decode_sched(B, n, C, num_sms);
    const TileCtas tc = tile_ctas(s);
    const int seg_max = decode_seg_max(s, tc);
    CUtensorMap tx, tw;
    const int wrows = split ? 2 * N : N;
    if (!make_tmap(&tx, X, static_cast<uint64_t>(K), static_cast<uint64_t>(B), kBM) ||
        !make_tmap(&tw, phi_t, static_cast<uint64_t>(K), static_cast<uint64_t>(wrows),
                   static_cast<uint32_t>((wrows + 15) / 16 * 16)))
        return cudaErrorInvalidValue;
    unsigned long long *bar = static_cast<unsigned long long *>(workspace);
    float *partials = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + kBarBytes);
    const unsigned long long epoch = next_epoch();
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    const uint32_t target = static_cast<uint32_t>(s.grid + (barrier_extra > 0 ? barrier_extra : 0));
    switch (n) {
#define MHC_CASE(k)                                                                            \
    case k:                                                                                    \
        return split ? launch_n<k, true>(tx, tw, X, B, C, s, tc, seg_max, a_pre, a_post, a_res, \
                                         bias, iters, Y, r, H_pre, H_post, H_res, F_pre,       \
                                         F_out, X_next, partials, bar, epoch, target,          \
                                         wait_limit_ns, device, stream)                        \
                     : launch_n<k, false>(tx, tw, X, B, C, s, tc, seg_max, a_pre, a_post,      \
                                          a_res, bias, iters, Y, r, H_pre, H_post, H_res,      \
                                          F_pre, F_out, X_next, partials, bar, epoch, target,  \
                                          wait_limit_ns, device, stream);
        MHC_CASE(1) MHC_CASE(2) MHC_CASE(3) MHC_CASE(4) MHC_CASE(5) MHC_CASE(6) MHC_CASE(7)
        MHC_CASE(8)
#undef MHC_CASE
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t read_and_clear_decode_status(int *status)
{
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    int v = 0, zero = 0;
    if ((e = cudaMemcpyFromSymbol(&v, g_decode_status, sizeof v)) != cudaSuccess) return e;
    if ((e = cudaMemcpyToSymbol(g_decode_status, &zero, sizeof zero)) != cudaSuccess) return e;
    *status = v;
    return cudaSuccess;
}

}  // namespace mhc
