// Step 1 of the mHC forward: the skinny projection GEMM fused with the RMS
// reduction (page "mHC 算法分析 & cutile 高效实现", §2.1, §2.2, fusion §3.1;
// split-K motivation §5.1).
//
//   Y[b][k] = Σ_q X[b][q]·φ[q][k]    r[b] = sqrt(Σ_q X[b][q]² / K)
//
// Design (sm_103a):
//   * Work unit = one 128-token × 64-K block (one pipeline stage; 2 or 4
//     boxes per stage measured no faster on GB300).  Units are ordered tile-major
//     (all K blocks of token tile 0, then tile 1, ...) and split into equal
//     contiguous ranges, one per persistent CTA (stream-K), so every SM gets
//     the same number of units whatever B and K are.  N is tiny (24 or 80),
//     so output tiling alone would leave most SMs idle (§5.1).
//   * Warp 0 (TMA), warp 1 (tcgen05.mma into TMEM) and warps 2-5 (Σx² from the
//     same shared-memory tiles, so X is read from HBM once) are the pipeline
//     of gemm_pipeline.cuh.  Warps 6-9 run the epilogue (tcgen05.ld of the
//     accumulator, partial sums, the fixed-order reduction), so the stage
//     consumers never wait on epilogue work.
//   * A tile covered by several CTAs is finished by the last one to arrive
//     (atomic ticket): it adds the partial sums in contributor order, so
//     the result is bitwise reproducible (§5.2 sums the splits in a fixed
//     order too).
//   * Every mbarrier wait is bounded; on expiry the CTA raises the device
//     status word, drains what it started, frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "check.cuh"
#include "gemm_pipeline.cuh"
#include "mhc_internal.h"
#include "mix.cuh"
#include "ptx.cuh"

namespace mhc {
namespace {

using pipe::kBK;
using pipe::kBM;
using pipe::Segment;
using pipe::Sched;
using pipe::SegIter;

constexpr int kThreads = 320;  // 10 warps: TMA, MMA, 4 × square-sum, 4 × epilogue
constexpr int kEpiThreads = 128;
constexpr int kReduceItems = 16;  // outputs per thread per round of the fixed-order sum
constexpr int kReduceBatch = 4;   // contributors loaded per batch: 64 loads in flight
constexpr int kRingBudget = 200 * 1024;
// columns of a row that the final segment's shared-memory sum takes at once
constexpr int kSumCols = 16;

__device__ int g_device_status;

template <int NPAD>
struct KCfg {
    using C = pipe::Cfg<NPAD, kRingBudget>;
    static constexpr int kSmemBytes = 1024 + C::kRingBytes + pipe::kSsBytes + pipe::kBarrierBytes;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

// Steps 2 and 3 for the token of one finished row (CoefArgs): n is fixed by
// the kernel's MMA width for all but a few (NPAD 16: n = 1, 2, 3; 48: n = 5,
// 6), so only the n whose width matches are compiled in.
template <int NPAD, bool kSplit, int nn>
constexpr bool kWidthOf = ((kSplit ? 2 : 1) * (nn * nn + 2 * nn) + 15) / 16 * 16 == NPAD;

template <int NPAD, bool kSplit, int nn>
__device__ __forceinline__ void row_coeffs_n(const CoefArgs &cf, const float *y, float rb,
                                             int64_t t)
{
    if constexpr (kWidthOf<NPAD, kSplit, nn>) {
        if (cf.n == nn) {
            float hp[nn], hq[nn], m[nn][nn];
            token_coeffs<nn>(y, rb, cf.bias, cf.a_pre, cf.a_post, cf.a_res, cf.iters, hp, hq, m);
            store_token_coeffs<nn>(t, hp, hq, m, cf.H_pre, cf.H_post, cf.H_res);
        }
    }
}

template <int NPAD, bool kSplit>
__device__ __forceinline__ void row_coeffs(const CoefArgs &cf, const float *y, float rb, int64_t t)
{
    row_coeffs_n<NPAD, kSplit, 1>(cf, y, rb, t);
    row_coeffs_n<NPAD, kSplit, 2>(cf, y, rb, t);
    row_coeffs_n<NPAD, kSplit, 3>(cf, y, rb, t);
    row_coeffs_n<NPAD, kSplit, 4>(cf, y, rb, t);
    row_coeffs_n<NPAD, kSplit, 5>(cf, y, rb, t);
    row_coeffs_n<NPAD, kSplit, 6>(cf, y, rb, t);
    row_coeffs_n<NPAD, kSplit, 7>(cf, y, rb, t);
    row_coeffs_n<NPAD, kSplit, 8>(cf, y, rb, t);
}

// The same for a pair of adjacent lanes (lane parity = half), each taking
// half of the token's rows; every lane of the warp calls it.
template <int NPAD, bool kSplit, int nn>
__device__ __forceinline__ void pair_coeffs_n(const CoefArgs &cf, const float *y, float rb,
                                              int half, bool store, int64_t t)
{
    if constexpr (kWidthOf<NPAD, kSplit, nn>) {
        if (cf.n == nn) {
            if constexpr (nn == 1) {
                if (store && half == 0) {
                    float hp[1], hq[1], m[1][1];
                    token_coeffs<1>(y, rb, cf.bias, cf.a_pre, cf.a_post, cf.a_res, cf.iters, hp,
                                    hq, m);
                    store_token_coeffs<1>(t, hp, hq, m, cf.H_pre, cf.H_post, cf.H_res);
                }
            } else {
                token_coeffs_pair<nn>(y, rb, cf.bias, cf.a_pre, cf.a_post, cf.a_res, cf.iters,
                                      half, store, t, cf.H_pre, cf.H_post, cf.H_res);
            }
        }
    }
}

// Coefficients of rows [64·g, 64·g + 64) of a finished tile whose rows (Ỹ then
// Σx², pitch rs floats) sit in shared memory, on the 128 threads gt of group
// g: a token per pair of lanes.  A lane past the tile's last row works on row
// 0 and stores nothing.
template <int NPAD, bool kSplit>
__device__ __forceinline__ void tile_coeffs_share(const CoefArgs &cf, const float *rowbuf, int rs,
                                                  int N, int K, int64_t row0, int rows, int64_t B,
                                                  int g, int gt)
{
    const int tk = g * 64 + (gt >> 1);
    const bool live = tk < rows && in_range(409, row0 + tk, 1, B);
    const float *yr = rowbuf + (live ? tk : 0) * rs;
    const float rb = sqrtf(yr[N] / static_cast<float>(K));
#define MHC_PAIR(k) pair_coeffs_n<NPAD, kSplit, k>(cf, yr, rb, gt & 1, live, row0 + tk);
    MHC_PAIR(1) MHC_PAIR(2) MHC_PAIR(3) MHC_PAIR(4) MHC_PAIR(5) MHC_PAIR(6) MHC_PAIR(7) MHC_PAIR(8)
#undef MHC_PAIR
}

// kSplit: the weight operand holds every column twice, as the bf16 value
// nearest the fp32 weight and the bf16 value nearest the remainder (rows 2k,
// 2k+1 of φᵀ), and the epilogue adds each pair: Ỹ[k] = acc[2k] + acc[2k+1].
// kFp8: X and φᵀ are e4m3 codes (128 per 128-byte row, kind::f8f6f4 MMAs).
template <int NPAD, bool kSplit, bool kFp8 = false>
__global__ void __launch_bounds__(kThreads, 1)
gemm_rms_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                int64_t B, int N, int K, Sched sch, float *__restrict__ Y, float *__restrict__ r,
                int *__restrict__ tile_tickets, float *__restrict__ partials,
                uint64_t wait_limit_ns, int64_t stall_stage, CoefArgs cf)
{
    using C = typename KCfg<NPAD>::C;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    pipe::Pipe p;
    pipe::carve<NPAD, kRingBudget>(p, smem, &g_device_status, wait_limit_ns);
    uint64_t *epi_bar = p.extra;      // epilogue group barrier
    uint64_t *red_bar = p.extra + 1;   // [2]: a chunk of the final segment's partials landed
    uint64_t *coef_bar = p.extra + 3;  // the final tile's rows are in shared memory
    volatile int *is_last = p.abort + 1;
    volatile int *coef_tile = p.abort + 2;  // 1 + that tile, or 0: no coefficients to help with

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;

    if (threadIdx.x == 0) {
        pipe::init_barriers(p);
        ptx::mbar_init(epi_bar, kEpiThreads);
        ptx::mbar_init(red_bar, 1);
        ptx::mbar_init(red_bar + 1, 1);
        ptx::mbar_init(coef_bar, kEpiThreads);
        *is_last = 0;
        *coef_tile = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tm_x);
        ptx::prefetch_tensormap(&tm_w);
    }
    if (warp == 1) ptx::tmem_alloc<C::kTmemCols>(p.tmem_holder);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    p.tmem_base = *p.tmem_holder;
    // everything above is on-chip set-up; global memory is touched only after
    // the previous kernel in the stream has completed
    ptx::pdl_wait();

    const SegIter segs{sch.lo(cta), sch.lo(cta + 1), sch.kbt};

    if (warp == 0) {
        if (lane == 0)  // X streams through once: evict it first
            pipe::producer<NPAD, SegIter, kFp8>(p, segs, &tm_x, &tm_w, ptx::policy_evict_first(),
                                                cta == 0 ? stall_stage : -1);
    } else if (warp == 1) {
        if (lane == 0) pipe::mma_issuer<NPAD, SegIter, kFp8>(p, segs);
    } else if (warp < 6) {
        pipe::square_sum<NPAD, SegIter, kFp8>(p, segs, (warp - 2) * 32 + lane, lane);
        // then the second half of the last tile's coefficients, when this CTA
        // finishes a tile in its last segment (the epilogue takes the first)
        // a warp helps only if all its lanes saw the tile (the pair shuffles)
        if (cf.H_pre && __all_sync(0xffffffffu, pipe::wait(p, coef_bar, 0))) {
            const int m1 = *coef_tile;
            if (m1 > 0) {
                const int64_t row0 = static_cast<int64_t>(m1 - 1) * kBM;
                const int rows = static_cast<int>((B - row0) < kBM ? (B - row0) : kBM);
                tile_coeffs_share<NPAD, kSplit>(cf, reinterpret_cast<const float *>(p.stages),
                                                (N + 1) | 1, N, K, row0, rows, B, 1,
                                                threadIdx.x - 64);
            }
        }
    } else {
        // ----------------------------------------------- epilogue (warps 6..9)
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        const int et = threadIdx.x - 192;  // 0..127 within the epilogue group
        uint32_t epi_phase = 0;
        int seg = 0;
        bool coef_arrived = false;  // each epilogue thread arrives on coef_bar once
        SegIter it = segs;
        Segment sg;
        while (it.next(sg)) {
            const int64_t row0 = static_cast<int64_t>(sg.m) * kBM;
            const int64_t grow = row0 + row;
            const bool whole = sg.k0 == 0 && sg.k1 == sch.kbt;
            const int stride = N + 1;
            // a partial is column-major, [N + 1][kBM]: stores and loads coalesce
            float *mine = partials + static_cast<int64_t>(cta + sg.m) * kBM * stride;
            const int slots = sch.grid + sch.m_tiles;  // partial slots of the workspace
            if (!whole && !in_range(401, cta + sg.m, 1, slots)) break;
            float ss;
            if constexpr (kSplit) {
                // chunks of 32 accumulator columns = 16 weight columns
                const bool ok = pipe::take_accumulator_chunked<NPAD>(
                    p, seg, q, lane, ss, [&](int c, const float (&v)[32]) {
                        if (grow >= B) return;
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int j = c * 16 + e;
                            if (j >= N) continue;
                            const float y = v[2 * e] + v[2 * e + 1];
                            if (whole)
                                Y[grow * N + j] = y;
                            else
                                mine[j * kBM + row] = y;
                        }
                    });
                if (!ok) break;
                ++seg;
                if (whole) {
                    if (grow < B) {
                        const float rr = sqrtf(ss / static_cast<float>(K));
                        r[grow] = rr;
                        // this thread's own stores of the row, read back
                        if (cf.H_pre) row_coeffs<NPAD, kSplit>(cf, Y + grow * N, rr, grow);
                    }
                    continue;
                }
                if (grow < B) mine[N * kBM + row] = ss;
            } else {
                float v[NPAD];
                if (!pipe::take_accumulator<NPAD>(p, seg, q, lane, v, ss)) break;
                ++seg;
                if (whole) {
                    // the whole K range of this tile is ours: write the result
                    if (grow < B) {
                        float *y = Y + grow * N;
#pragma unroll
                        for (int j = 0; j < NPAD; ++j)
                            if (j < N) y[j] = v[j];
                        const float rr = sqrtf(ss / static_cast<float>(K));
                        r[grow] = rr;
                        if (cf.H_pre) row_coeffs<NPAD, kSplit>(cf, v, rr, grow);
                    }
                    continue;
                }
                // partial: park it in this (cta, tile) slot, then take a ticket
                if (grow < B) {
#pragma unroll
                    for (int j = 0; j < NPAD; ++j)
                        if (j < N) mine[j * kBM + row] = v[j];
                    mine[N * kBM + row] = ss;
                }
            }
            // the finishing CTA may read this partial by bulk copy (the async
            // proxy): order the generic stores for that proxy too, then release
            asm volatile("fence.proxy.async.global;" ::: "memory");
            __threadfence();
            if (!pipe::group_sync(p, epi_bar, epi_phase)) break;
            const int first = sch.owner(static_cast<int64_t>(sg.m) * sch.kbt);
            const int last = sch.owner(static_cast<int64_t>(sg.m + 1) * sch.kbt - 1);
            // the tile's ticket and its contributors' slots first + m .. last + m
            if (!in_range(402, sg.m, 1, sch.m_tiles) ||
                !in_range(403, first + sg.m, last - first + 1, slots))
                break;
            if (et == 0) {
                const int prev = atomicAdd(&tile_tickets[sg.m], 1);
                *is_last = (prev == last - first);
            }
            if (!pipe::group_sync(p, epi_bar, epi_phase)) break;
            if (*is_last) {
                __threadfence();
                const int rows = static_cast<int>((B - row0) < kBM ? (B - row0) : kBM);
                const int items = kBM * stride;  // item i: column i / kBM, row i % kBM
                const float *p0 = partials + static_cast<int64_t>(first + sg.m) * kBM * stride;
                const int64_t slot_stride = static_cast<int64_t>(kBM) * stride;
                const int nc = last - first + 1;
                SegIter peek = it;
                Segment nx;
                // This CTA's last segment: its stage ring is idle (every stage has been
                // consumed).  The contributors' partials come into it by bulk copies, a
                // chunk of columns of every contributor at a time, two chunks in
                // flight; loads into registers would take one round trip per batch of
                // contributors, and this sum ends the kernel on the critical path.
                const int rs = stride | 1;  // odd row pitch: the row writes miss no bank
                const uint32_t row_bytes = static_cast<uint32_t>(kBM) * rs * 4;
                const int64_t room = (C::kRingBytes - static_cast<int64_t>(row_bytes)) / 2;
                const int cc = static_cast<int>(
                    min(static_cast<int64_t>(stride), room / (static_cast<int64_t>(nc) * kBM * 4)));
                if (!peek.next(nx) && cc > 0) {
                    float *rowbuf = reinterpret_cast<float *>(p.stages);  // [kBM][rs]
                    float *const chunk0 = rowbuf + kBM * rs;  // two buffers, [nc][cc][kBM]
                    const int64_t half = static_cast<int64_t>(nc) * cc * kBM;
                    if (!in_range(404, 0, kBM * rs + 2 * half, C::kRingBytes / 4)) break;
                    const int nchunks = (stride + cc - 1) / cc;
                    auto issue = [&](int k) {
                        const int c0 = k * cc;
                        const int w = min(cc, stride - c0);
                        if (!in_range(405, c0, w, stride)) return;  // its wait then runs out
                        const uint32_t bytes = static_cast<uint32_t>(w) * kBM * 4;
                        ptx::mbar_arrive_expect_tx(red_bar + (k & 1), bytes * nc);
                        for (int c = 0; c < nc; ++c)
                            ptx::bulk_load(chunk0 + (k & 1) * half + static_cast<int64_t>(c) * cc * kBM,
                                           p0 + c * slot_stride + static_cast<int64_t>(c0) * kBM,
                                           bytes, red_bar + (k & 1), ptx::policy_evict_first());
                    };
                    if (et == 0) {
                        // the partials were written through the generic proxy
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                        issue(0);
                        if (nchunks > 1) issue(1);
                    }
                    bool ok = true;
                    int k = 0;
                    for (; k < nchunks; ++k) {
                        if (!pipe::wait(p, red_bar + (k & 1), (k >> 1) & 1)) {
                            ok = false;
                            break;
                        }
                        // thread et: row et, its contributors in order as in the
                        // general path below, so the sums agree to the bit
                        if (et < rows) {
                            const float *buf = chunk0 + (k & 1) * half + et;
                            const int c0 = k * cc;
                            const int w = min(cc, stride - c0);
                            // kSumCols columns at once: their loads are independent
                            for (int col0 = 0; col0 < w; col0 += kSumCols) {
                                float acc[kSumCols];
#pragma unroll
                                for (int u = 0; u < kSumCols; ++u) acc[u] = 0.f;
#pragma unroll 2
                                for (int c = 0; c < nc; ++c) {
                                    const float *src = buf + (static_cast<int64_t>(c) * cc + col0) * kBM;
                                    float v[kSumCols];
#pragma unroll
                                    for (int u = 0; u < kSumCols; ++u)
                                        v[u] = col0 + u < w ? src[u * kBM] : 0.f;
#pragma unroll
                                    for (int u = 0; u < kSumCols; ++u) acc[u] += v[u];
                                }
#pragma unroll
                                for (int u = 0; u < kSumCols; ++u)
                                    if (col0 + u < w) rowbuf[et * rs + c0 + col0 + u] = acc[u];
                            }
                        }
                        // every read of this chunk's buffer is done before it refills
                        if (!pipe::group_sync(p, epi_bar, epi_phase)) {
                            ok = false;
                            break;
                        }
                        if (et == 0 && k + 2 < nchunks) issue(k + 2);
                    }
                    if (!ok) {
                        // the copies issued land before the CTA may exit
                        volatile int never = 0;
                        for (int j = k; j < nchunks && j < k + 2; ++j)
                            ptx::mbar_wait_bounded(red_bar + (j & 1), (j >> 1) & 1, &never,
                                                   p.limit_ns);
                        break;
                    }
                    // The tile's rows of Y are contiguous (and 16-byte aligned: row0 is
                    // a multiple of 128): 16-byte stores, each thread's (row, column)
                    // stepped along without a division.  N >= 3, so one wrap suffices.
                    {
                        float *yt = Y + row0 * N;
                        const int total = rows * N, quads = total >> 2;
                        const int srow = 4 * kEpiThreads / N, scol = 4 * kEpiThreads % N;
                        int yr = 4 * et / N, yc = 4 * et % N;
                        for (int q4 = et; q4 < quads; q4 += kEpiThreads) {
                            if (!in_range(406, row0 * N + 4 * q4, 4, B * N)) break;
                            float f[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const bool wrap = yc + u >= N;
                                f[u] = rowbuf[(yr + wrap) * rs + yc + u - (wrap ? N : 0)];
                            }
                            *reinterpret_cast<float4 *>(yt + 4 * q4) = make_float4(f[0], f[1], f[2], f[3]);
                            yc += scol;
                            yr += srow;
                            if (yc >= N) {
                                yc -= N;
                                ++yr;
                            }
                        }
                        for (int i = 4 * quads + et; i < total; i += kEpiThreads)
                            yt[i] = rowbuf[(i / N) * rs + i % N];
                    }
                    if (et < rows) r[row0 + et] = sqrtf(rowbuf[et * rs + N] / static_cast<float>(K));
                    if (et == 0) tile_tickets[sg.m] = 0;
                    if (cf.H_pre) {
                        // the square-sum warps, idle now, take rows 64..127
                        if (et == 0) *coef_tile = static_cast<int>(sg.m) + 1;
                        ptx::mbar_arrive(coef_bar);
                        coef_arrived = true;
                        tile_coeffs_share<NPAD, kSplit>(cf, rowbuf, rs, N, K, row0, rows, B, 0, et);
                    }
                    continue;
                }
                // fixed-order sum over the contributors first..last: a batch of
                // contributors x items is loaded before it is added, in order
                for (int i0 = et; i0 < items; i0 += kEpiThreads * kReduceItems) {
                    float acc_s[kReduceItems];
#pragma unroll
                    for (int u = 0; u < kReduceItems; ++u) acc_s[u] = 0.f;
                    for (int c0 = 0; c0 < nc; c0 += kReduceBatch) {
                        float vb[kReduceBatch][kReduceItems];
#pragma unroll
                        for (int c = 0; c < kReduceBatch; ++c)
#pragma unroll
                            for (int u = 0; u < kReduceItems; ++u) {
                                const int i = i0 + u * kEpiThreads;
                                vb[c][u] = (c0 + c < nc && i < items && i % kBM < rows)
                                               ? __ldcg(p0 + (c0 + c) * slot_stride + i)
                                               : 0.f;  // acc + 0 is exact: acc is never -0
                            }
#pragma unroll
                        for (int c = 0; c < kReduceBatch; ++c)
#pragma unroll
                            for (int u = 0; u < kReduceItems; ++u) acc_s[u] += vb[c][u];
                    }
#pragma unroll
                    for (int u = 0; u < kReduceItems; ++u) {
                        const int i = i0 + u * kEpiThreads;
                        if (i >= items) break;
                        const int rr = i % kBM, cc = i / kBM;
                        if (rr >= rows) continue;
                        if (cc < N)
                            Y[(row0 + rr) * N + cc] = acc_s[u];
                        else
                            r[row0 + rr] = sqrtf(acc_s[u] / static_cast<float>(K));
                    }
                }
                // thread et wrote all of row et (i % 128 == et): its coefficients
                if (cf.H_pre && et < rows)
                    row_coeffs<NPAD, kSplit>(cf, Y + (row0 + et) * N, r[row0 + et], row0 + et);
                if (et == 0) tile_tickets[sg.m] = 0;
            }
        }
        if (!coef_arrived) ptx::mbar_arrive(coef_bar);  // nothing to help with
    }

    // lane 0 of the TMA and MMA warps ran alone: reconverge every warp before
    // the CTA barrier, which needs whole warps
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    // Let the next kernel launch only now: CTAs of a dependent kernel that sit
    // resident in pdl_wait next to this one for its whole run slow it down
    // (measured: +13% at B=16384), while a trigger at the end still hides
    // the launch latency.
    ptx::pdl_trigger();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc<C::kTmemCols>(p.tmem_base);
    }
}

// Clears the tile tickets of a call before its GEMM kernel runs.
__global__ void zero_tickets_kernel(int *tickets, int count)
{
    ptx::pdl_wait();
    ptx::pdl_trigger();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < count; i += gridDim.x * blockDim.x)
        tickets[i] = 0;
}

// ------------------------------------------------------------------ host

// Grid: one CTA per SM, but no more than 32 contributors per token tile (the
// last arriver's fixed-order sum grows with the fan-in) and at least one
// stage of K per CTA.
Sched make_sched(int64_t B, int n, int64_t C, int num_sms, int k_per_block = kBK)
{
    Sched s;
    s.m_tiles = static_cast<int>((B + kBM - 1) / kBM);
    s.kbt = static_cast<int>((n * C + k_per_block - 1) / k_per_block);
    s.total = static_cast<int64_t>(s.m_tiles) * s.kbt;
    int64_t g = num_sms;
    if (g > 32LL * s.m_tiles) g = 32LL * s.m_tiles;
    if (g > s.total) g = s.total;
    if (g < 1) g = 1;
    s.grid = static_cast<int>(g);
    return s;
}

size_t tickets_bytes(int m_tiles) { return (static_cast<size_t>(m_tiles) * 4 + 255) / 256 * 256; }

struct LaunchArgs {
    const CUtensorMap *tx, *tw;
    int64_t B;
    int N, K;
    Sched s;
    float *Y, *r;
    int *tickets;
    float *partials;
    cudaStream_t stream;
    int device;
    uint64_t wait_limit_ns;
    int64_t stall_stage;
    CoefArgs coef;
};

template <int NPAD, bool kSplit, bool kFp8 = false>
cudaError_t launch_cfg(const LaunchArgs &a)
{
    using Cf = KCfg<NPAD>;
    static uint64_t configured = 0;  // one bit per device
    static std::mutex mu;
    if (a.device < 64 && !((configured >> a.device) & 1)) {
        std::lock_guard<std::mutex> lock(mu);
        cudaError_t e = cudaFuncSetAttribute(gemm_rms_kernel<NPAD, kSplit, kFp8>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Cf::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured |= 1ull << a.device;
    }
    return launch_pdl(gemm_rms_kernel<NPAD, kSplit, kFp8>, dim3(a.s.grid), dim3(kThreads),
                      Cf::kSmemBytes, a.stream, *a.tx, *a.tw, a.B, a.N, a.K, a.s, a.Y, a.r,
                      a.tickets, a.partials, a.wait_limit_ns, a.stall_stage, a.coef);
}

cudaError_t dispatch(int npad, bool split, bool fp8, const LaunchArgs &a)
{
    if (fp8) {
        switch (npad) {
        case 16: return launch_cfg<16, false, true>(a);
        case 32: return launch_cfg<32, false, true>(a);
        case 48: return launch_cfg<48, false, true>(a);
        case 64: return launch_cfg<64, false, true>(a);
        case 80: return launch_cfg<80, false, true>(a);
        default: return cudaErrorInvalidValue;
        }
    }
    if (split) {
        switch (npad) {  // 2N padded: n = 1, 2 -> 16; 3 -> 32; 4 -> 48; 5 -> 80; 6 -> 96; 7 -> 128; 8 -> 160
        case 16: return launch_cfg<16, true>(a);
        case 32: return launch_cfg<32, true>(a);
        case 48: return launch_cfg<48, true>(a);
        case 80: return launch_cfg<80, true>(a);
        case 96: return launch_cfg<96, true>(a);
        case 128: return launch_cfg<128, true>(a);
        case 160: return launch_cfg<160, true>(a);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (npad) {
    case 16: return launch_cfg<16, false>(a);
    case 32: return launch_cfg<32, false>(a);
    case 48: return launch_cfg<48, false>(a);
    case 64: return launch_cfg<64, false>(a);
    case 80: return launch_cfg<80, false>(a);
    default: return cudaErrorInvalidValue;
    }
}

// Splits an fp32 φᵀ [N][K] into bf16 rows 2k (the bf16 value nearest φ) and
// 2k+1 (the bf16 value nearest the remainder φ - hi).
__global__ void split_phi_kernel(const float *__restrict__ phi_t, int64_t N, int64_t K,
                                 uint16_t *__restrict__ out)
{
    ptx::pdl_wait();
    ptx::pdl_trigger();
    const int64_t total = N * K;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t k = i / K, q = i - k * K;
        if (!in_range(407, 2 * k + 1, 1, 2 * N)) break;
        const float v = phi_t[i];
        const uint32_t hi2 = pack_bf16_rn(v, 0.f);
        const float hi = __uint_as_float(hi2 << 16);
        const uint32_t lo2 = pack_bf16_rn(v - hi, 0.f);
        out[(2 * k) * K + q] = static_cast<uint16_t>(hi2 & 0xFFFFu);
        out[(2 * k + 1) * K + q] = static_cast<uint16_t>(lo2 & 0xFFFFu);
    }
}

}  // namespace

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

static bool make_tmap_2d(CUtensorMap *m, CUtensorMapDataType type, int esize, const void *base,
                         uint64_t cols, uint64_t rows, uint32_t box_rows)
{
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * static_cast<uint64_t>(esize)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esize), box_rows};  // one 128-byte row
    cuuint32_t estr[2] = {1, 1};
    return f(m, type, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 tensor [rows][cols] (cols contiguous), box [box_rows][64], 128-byte swizzle.
bool make_tmap(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_rows)
{
    return make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, cols, rows, box_rows);
}

// The same for e4m3 codes: box [box_rows][128].
static bool make_tmap_e4m3(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows,
                           uint32_t box_rows)
{
    return make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, cols, rows, box_rows);
}

size_t gemm_rms_workspace_bytes(int64_t B, int n, int64_t C, int num_sms)
{
    if (B <= 0) return 0;
    const Sched s = make_sched(B, n, C, num_sms);
    const int N = num_coeffs(n);
    const size_t slots = static_cast<size_t>(s.grid) + s.m_tiles;
    return tickets_bytes(s.m_tiles) + slots * kBM * (N + 1) * sizeof(float);
}

static cudaError_t launch_gemm_rms_impl(const void *X, const void *phi_t, int64_t B, int n,
                                        int64_t C, float *Y, float *r, void *workspace,
                                        int num_sms, cudaStream_t stream, uint64_t wait_limit_ns,
                                        int64_t stall_stage, bool split, bool fp8,
                                        const CoefArgs &coef)
{
    const int N = num_coeffs(n);
    const int64_t K = n * C;
    const Sched s = make_sched(B, n, C, num_sms, fp8 ? 2 * kBK : kBK);
    CUtensorMap tx, tw;
    const int wrows = split ? 2 * N : N;  // rows of the weight operand
    const int npad = (wrows + 15) / 16 * 16;
    const auto tmap = fp8 ? make_tmap_e4m3 : make_tmap;
    if (!tmap(&tx, X, static_cast<uint64_t>(K), static_cast<uint64_t>(B), kBM) ||
        !tmap(&tw, phi_t, static_cast<uint64_t>(K), static_cast<uint64_t>(wrows),
              static_cast<uint32_t>(npad)))
        return cudaErrorInvalidValue;
    int *tickets = static_cast<int *>(workspace);
    float *partials = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                                tickets_bytes(s.m_tiles));
    const int zero_blocks = s.m_tiles < 256 * 64 ? (s.m_tiles + 255) / 256 : 64;
    cudaError_t e = launch_pdl(zero_tickets_kernel, dim3(zero_blocks), dim3(256), 0, stream,
                               tickets, s.m_tiles);
    if (e != cudaSuccess) return e;
    int device = 0;
    if ((e = cudaGetDevice(&device)) != cudaSuccess) return e;
    const LaunchArgs a{&tx, &tw, B, N, static_cast<int>(K), s, Y, r, tickets, partials, stream,
                       device, wait_limit_ns, stall_stage, coef};
    return dispatch(npad, split, fp8, a);
}

cudaError_t launch_gemm_rms(const uint16_t *X, const uint16_t *phi_t, int64_t B, int n,
                            int64_t C, float *Y, float *r, void *workspace, int num_sms,
                            cudaStream_t stream, uint64_t wait_limit_ns, int64_t stall_stage,
                            const CoefArgs &coef)
{
    return launch_gemm_rms_impl(X, phi_t, B, n, C, Y, r, workspace, num_sms, stream,
                                wait_limit_ns, stall_stage, false, false, coef);
}

cudaError_t launch_gemm_rms_split(const uint16_t *X, const uint16_t *phi_split, int64_t B, int n,
                                  int64_t C, float *Y, float *r, void *workspace, int num_sms,
                                  cudaStream_t stream, const CoefArgs &coef)
{
    return launch_gemm_rms_impl(X, phi_split, B, n, C, Y, r, workspace, num_sms, stream,
                                kWaitLimitNs, -1, true, false, coef);
}

cudaError_t launch_gemm_rms_e4m3(const uint8_t *X, const uint8_t *phi_t, int64_t B, int n,
                                 int64_t C, float *Y, float *r, void *workspace, int num_sms,
                                 cudaStream_t stream, const CoefArgs &coef)
{
    return launch_gemm_rms_impl(X, phi_t, B, n, C, Y, r, workspace, num_sms, stream,
                                kWaitLimitNs, -1, false, true, coef);
}

cudaError_t launch_split_phi(const float *phi_t, int n, int64_t C, uint16_t *phi_split,
                             cudaStream_t stream)
{
    const int64_t N = num_coeffs(n), K = n * C;
    const int64_t need = (N * K + 255) / 256;
    const int blocks = static_cast<int>(need < 4096 ? need : 4096);
    return launch_pdl(split_phi_kernel, dim3(blocks), dim3(256), 0, stream, phi_t, N, K,
                      phi_split);
}

cudaError_t read_and_clear_device_status(int *status)
{
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    int v = 0, zero = 0;
    if ((e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof v)) != cudaSuccess) return e;
    if ((e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero)) != cudaSuccess) return e;
    *status = v;
    return cudaSuccess;
}

}  // namespace mhc
