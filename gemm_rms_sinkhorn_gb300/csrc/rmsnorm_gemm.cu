// C = rmsnorm(A) @ B with the normalisation folded into the GEMM as the page
// "Towards Free Normalization: Fusing Normalization into GEMM and Attention
// Kernels" (PyTorch blog), §2 "Lazy Pre-Norm", describes it:
//
//   rstd[m] = 1 / sqrt(Σ_q A[m][q]² / K + eps)
//   C[m][n] = (Σ_q A[m][q]·B[q][n]) · rstd[m]        ((A·rstd) @ B = (A @ B)·rstd)
//
// The row sum of squares is reduced from the same shared-memory tiles the
// tensor cores consume, by separate warps, so A leaves HBM once and the
// normalisation costs no pass of its own; the scaling by rstd is the
// epilogue.  It reuses the pipeline of gemm_pipeline.cuh (the mHC GEMM+RMS is
// the skinny case of this computation) with a column-tile dimension:
//
//   tiles    128 rows × NT columns of C, NT = 32, 64, 128 or 256 by N, row
//            tiles outermost so a CTA's consecutive tiles share their A rows;
//   schedule with at least one tile per CTA, every CTA owns a contiguous run
//            of whole tiles (no partial sums); with fewer tiles than CTAs the
//            K blocks are split stream-K as in gemm_rms.cu, and the last CTA
//            to finish a tile adds the partials in contributor order;
//   epilogue the accumulator leaves TMEM 32 columns at a time, is scaled by
//            rstd, rounded to bf16 (RNE) and stored;
//   256 rows with 256-column tiles, long K and enough of them, a CTA takes
//            256 × 256 tiles in a grouped order that keeps the GPU on a few
//            row tiles at a time (see "256-row tiles" below).
// In the 128-row kernels the square sums of a row tile are computed once per
// run of its tiles in a CTA, not once per column tile as on the page: the
// CUDA-core work is cheap, but its shared-memory reads compete with the
// tensor cores' operand reads.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "check.cuh"
#include "gemm_pipeline.cuh"
#include "mhc_internal.h"
#include "ptx.cuh"

namespace mhc {
namespace {

using pipe::kBK;
using pipe::kBM;
using pipe::Segment;

constexpr int kThreads = 320;  // 10 warps: TMA, MMA, 4 × square-sum, 4 × epilogue
constexpr int kEpiThreads = 128;
constexpr int kRingBudget = 200 * 1024;
constexpr int kMaxFanIn = 32;  // contributors per tile when K is split

__device__ int g_rng_status;

template <int NT>
struct RCfg {
    using C = pipe::Cfg<NT, kRingBudget>;
    static constexpr int kRstdBytes = kBM * 4;  // the last arriver's rstd of each row
    static constexpr int kSmemBytes =
        1024 + C::kRingBytes + pipe::kSsBytes + pipe::kBarrierBytes + kRstdBytes;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

// Units (tile, K block), tile = row tile · n_tiles + column tile.  With
// aligned == 1 the ranges start and end on tile boundaries.
struct RSched {
    int64_t tiles, total;  // tiles; tiles · kbt units
    int kbt, n_tiles, grid, aligned;
    __host__ __device__ int64_t lo(int c) const {
        return aligned ? (tiles * c / grid) * kbt : total * c / grid;
    }
    __host__ __device__ int owner(int64_t u) const {  // CTA whose range holds unit u
        if (aligned) return static_cast<int>(((u / kbt + 1) * grid - 1) / tiles);
        return static_cast<int>(((u + 1) * grid - 1) / total);
    }
};

struct RIter {
    int64_t u, end;
    int kbt, n_tiles;
    __device__ bool next(Segment &s) {
        if (u >= end) return false;
        const int64_t t = u / kbt;
        s.m = static_cast<int>(t / n_tiles);
        s.n = static_cast<int>(t - static_cast<int64_t>(s.m) * n_tiles);
        s.k0 = static_cast<int>(u - t * kbt);
        const int64_t left = end - u;
        s.k1 = left < kbt - s.k0 ? s.k0 + static_cast<int>(left) : kbt;
        u += s.k1 - s.k0;
        return true;
    }
};

__device__ __forceinline__ RIter make_segs(const RSched &sch, int cta)
{
    return RIter{sch.lo(cta), sch.lo(cta + 1), sch.kbt, sch.n_tiles};
}

// Σa² of one 128-byte stage row (64 bf16) into four partial sums.
__device__ __forceinline__ void row_sq64(const uint8_t *arow, int row, float (&s)[4])
{
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        // chunk j of the row is at chunk j ^ (row % 8) (128-byte swizzle)
        const uint4 v = *reinterpret_cast<const uint4 *>(arow + ((j ^ (row & 7)) << 4));
        const float a0 = bf16_lo(v.x), a1 = bf16_hi(v.x), a2 = bf16_lo(v.y);
        const float a3 = bf16_hi(v.y), a4 = bf16_lo(v.z), a5 = bf16_hi(v.z);
        const float a6 = bf16_lo(v.w), a7 = bf16_hi(v.w);
        s[0] = fmaf(a0, a0, s[0]); s[1] = fmaf(a1, a1, s[1]);
        s[2] = fmaf(a2, a2, s[2]); s[3] = fmaf(a3, a3, s[3]);
        s[0] = fmaf(a4, a4, s[0]); s[1] = fmaf(a5, a5, s[1]);
        s[2] = fmaf(a6, a6, s[2]); s[3] = fmaf(a7, a7, s[3]);
    }
}

// As pipe::square_sum (bf16), but a whole tile whose row tile is that of the
// previous whole tile hands over the previous sum without reading its stages:
// the A rows, hence Σa², are the same.  Shared-memory reads are what bound
// this kernel (the TMA writes and the MMA operand reads share the port), so
// the redundant 16 KB read of every stage matters.  The stages are still
// waited for and released in order.
template <typename It>
__device__ void row_square_sums(const pipe::Pipe &p, It it, int kbt, int row, int lane)
{
    int stage = 0;
    uint32_t phase = 0;
    int seg = 0;
    int prev_m = -1;  // row tile of the previous whole tile
    float prev_ss = 0.f;
    Segment sg;
    bool ok = true;
    while (ok && it.next(sg)) {
        const bool whole = sg.k0 == 0 && sg.k1 == kbt;
        const bool reuse = whole && sg.m == prev_m;
        float ss[4] = {0.f, 0.f, 0.f, 0.f};
        for (int kb = sg.k0; kb < sg.k1; ++kb) {
            if (!pipe::wait(p, &p.full[stage], phase)) {
                ok = false;
                break;
            }
            if (!reuse) row_sq64(p.stages + stage * p.stage_bytes + row * 128, row, ss);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&p.empty[stage]);
            if (++stage == p.stages_n) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        const float sum = reuse ? prev_ss : (ss[0] + ss[1]) + (ss[2] + ss[3]);
        const int buf = seg & 1;
        if (!pipe::wait(p, &p.ss_empty[buf], ((seg >> 1) & 1) ^ 1)) break;
        p.ss_buf[buf * kBM + row] = sum;
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&p.ss_full[buf]);
        prev_m = whole ? sg.m : -1;
        prev_ss = sum;
        ++seg;
    }
}

// 32 accumulator columns of this thread's row, scaled and stored as bf16.
__device__ __forceinline__ void store_cols32(const float (&v)[32], float rstd, uint16_t *dst,
                                             int valid)
{
    float t[8];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        if (g * 8 >= valid) break;
#pragma unroll
        for (int e = 0; e < 8; ++e) t[e] = v[g * 8 + e] * rstd;
        const uint4 w = make_uint4(pack_bf16_rn(t[0], t[1]), pack_bf16_rn(t[2], t[3]),
                                   pack_bf16_rn(t[4], t[5]), pack_bf16_rn(t[6], t[7]));
        *reinterpret_cast<uint4 *>(dst + g * 8) = w;
    }
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 1)
rmsnorm_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                    const __grid_constant__ CUtensorMap tm_b, int64_t M, int64_t N, int K,
                    float eps, RSched sch, uint16_t *__restrict__ Cout, int *__restrict__ tickets,
                    float *__restrict__ partials, uint64_t wait_limit_ns)
{
    using Cf = typename RCfg<NT>::C;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    pipe::Pipe p;
    float *rstd_s = reinterpret_cast<float *>(
        pipe::carve<NT, kRingBudget>(p, smem, &g_rng_status, wait_limit_ns));
    uint64_t *epi_bar = p.extra;
    volatile int *is_last = p.abort + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;

    if (threadIdx.x == 0) {
        pipe::init_barriers(p);
        ptx::mbar_init(epi_bar, kEpiThreads);
        *is_last = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tm_a);
        ptx::prefetch_tensormap(&tm_b);
    }
    if (warp == 1) ptx::tmem_alloc<Cf::kTmemCols>(p.tmem_holder);
    ptx::tc_fence_before();
    __syncwarp();  // whole warps at the (aligned) barrier
    __syncthreads();
    ptx::tc_fence_after();
    p.tmem_base = *p.tmem_holder;
    ptx::pdl_wait();

    const auto segs = make_segs(sch, cta);
    const float inv_k = 1.0f / static_cast<float>(K);

    if (warp == 0) {
        if (lane == 0)  // A rows are re-read by the next column tiles: keep them in L2
            pipe::producer<NT>(p, segs, &tm_a, &tm_b, ptx::policy_evict_normal(), -1);
    } else if (warp == 1) {
        if (lane == 0) pipe::mma_issuer<NT>(p, segs);
    } else if (warp < 6) {
        row_square_sums(p, segs, sch.kbt, (warp - 2) * 32 + lane, lane);
    } else {
        // ----------------------------------------------- epilogue (warps 6..9)
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        const int et = threadIdx.x - 192;
        uint32_t epi_phase = 0;
        int seg = 0;
        auto it = segs;
        Segment sg;
        while (it.next(sg)) {
            const int acc = seg & 1;
            const uint32_t par = (seg >> 1) & 1;
            if (!pipe::wait(p, &p.acc_full[acc], par)) break;
            ptx::tc_fence_after();
            if (!pipe::wait(p, &p.ss_full[acc], par)) break;
            const float ss = p.ss_buf[acc * kBM + row];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&p.ss_empty[acc]);
            ++seg;

            const int64_t grow = static_cast<int64_t>(sg.m) * kBM + row;
            const int64_t col0 = static_cast<int64_t>(sg.n) * NT;
            const uint32_t taddr = p.tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * NT);
            const bool whole = sg.k0 == 0 && sg.k1 == sch.kbt;
            const int stride = NT + 1;
            const int64_t tile = static_cast<int64_t>(sg.m) * sch.n_tiles + sg.n;
            float *mine = partials + static_cast<int64_t>(cta + tile) * kBM * stride;
            const float rstd = whole ? rsqrtf(ss * inv_k + eps) : 0.f;
#pragma unroll 1
            for (int j = 0; j < NT / 32; ++j) {
                float v[32], t16[16];
                ptx::tmem_ld_16(taddr + j * 32, t16);
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = t16[e];
                ptx::tmem_ld_16(taddr + j * 32 + 16, t16);
#pragma unroll
                for (int e = 0; e < 16; ++e) v[16 + e] = t16[e];
                ptx::tmem_ld_wait();
                const int64_t c0 = col0 + j * 32;
                if (grow < M && c0 < N) {
                    if (whole) {
                        const int valid = N - c0 < 32 ? static_cast<int>(N - c0) : 32;
                        if (in_range(701, grow, 1, M) && in_range(702, c0, (valid + 7) / 8 * 8, N))
                            store_cols32(v, rstd, Cout + grow * N + c0, valid);
                    } else if (in_range(703, cta + tile, 1,
                                        static_cast<int64_t>(sch.grid) + sch.tiles)) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) mine[row * stride + j * 32 + e] = v[e];
                    }
                }
                __syncwarp();  // the next tcgen05.ld is warp-collective
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&p.acc_empty[acc]);
            if (whole) continue;

            // a partial: park the square sum too, take a ticket, and the last
            // contributor adds the partials in contributor order
            if (grow < M) mine[row * stride + NT] = ss;
            __threadfence();
            if (!pipe::group_sync(p, epi_bar, epi_phase)) break;
            const int first = sch.owner(tile * sch.kbt);
            const int last = sch.owner((tile + 1) * sch.kbt - 1);
            if (!in_range(704, tile, 1, sch.tiles) ||
                !in_range(705, first + tile, last - first + 1,
                          static_cast<int64_t>(sch.grid) + sch.tiles))
                break;
            if (et == 0) {
                const int prev = atomicAdd(&tickets[tile], 1);
                *is_last = (prev == last - first);
            }
            if (!pipe::group_sync(p, epi_bar, epi_phase)) break;
            if (!*is_last) continue;
            __threadfence();
            const int64_t row0 = static_cast<int64_t>(sg.m) * kBM;
            const int rows = static_cast<int>(M - row0 < kBM ? M - row0 : kBM);
            const int64_t slot_stride = static_cast<int64_t>(kBM) * stride;
            const float *p0 = partials + static_cast<int64_t>(first + tile) * slot_stride;
            const int nc = last - first + 1;
            // rstd of every row first (its square sums, in contributor order)
            if (et < rows) {
                float s = 0.f;
                for (int c = 0; c < nc; ++c) s += __ldcg(p0 + c * slot_stride + et * stride + NT);
                rstd_s[et] = rsqrtf(s * inv_k + eps);
            }
            if (!pipe::group_sync(p, epi_bar, epi_phase)) break;
            // then the columns: thread et sums and stores 8 consecutive columns of
            // one row (16-byte stores), rows × NT/8 items
            const int cols = static_cast<int>(N - col0 < NT ? N - col0 : NT);
            const int items = rows * (NT / 8);
            for (int i = et; i < items; i += kEpiThreads) {
                const int rr = i / (NT / 8), cc = (i - rr * (NT / 8)) * 8;
                if (cc >= cols) continue;
                if (!in_range(706, row0 + rr, 1, M) || !in_range(707, col0 + cc, 8, N)) continue;
                float a8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) a8[e] = 0.f;
                for (int c = 0; c < nc; ++c) {
                    const float *src = p0 + c * slot_stride + rr * stride + cc;
#pragma unroll
                    for (int e = 0; e < 8; ++e) a8[e] += __ldcg(src + e);
                }
                const float rs = rstd_s[rr];
                const uint4 w = make_uint4(pack_bf16_rn(a8[0] * rs, a8[1] * rs),
                                           pack_bf16_rn(a8[2] * rs, a8[3] * rs),
                                           pack_bf16_rn(a8[4] * rs, a8[5] * rs),
                                           pack_bf16_rn(a8[6] * rs, a8[7] * rs));
                *reinterpret_cast<uint4 *>(Cout + (row0 + rr) * N + col0 + cc) = w;
            }
            if (et == 0) tickets[tile] = 0;
            if (!pipe::group_sync(p, epi_bar, epi_phase)) break;  // rstd_s is reused
        }
    }

    // lane 0 of the TMA and MMA warps ran alone: reconverge every warp before
    // the CTA barrier, which needs whole warps
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::pdl_trigger();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc<Cf::kTmemCols>(p.tmem_base);
    }
}

// -------------------------------------------------------- 256-row tiles
// With 256-column tiles and at least as many 256-row tiles as SMs, a CTA
// takes 256 × 256 tiles: per K block one 256-row A box and one B box (64 KB),
// two M=128 MMAs sharing the B operand into two 256-column accumulators (all
// 512 TMEM columns).  That is 32 KB of stage per 4.2 MFLOP instead of 48, and
// the ring's bytes against L2 latency are what bound the 128-row kernel.  The
// accumulators are single-buffered: the epilogue frees the first as soon as it
// has read it, so the next tile's first MMAs overlap the second half.
//
// Tile order: groups of kGroup2 row tiles, column-major inside a group, dealt
// round-robin over the CTAs, so the 152 tiles in flight at any time span about
// kGroup2 + 2 row tiles (at K = 4096, 20 MB of A) next to the B boxes, which
// stay in L2.  A CTA's consecutive tiles then sit in different row tiles, so
// each tile computes its own square sums (the A stages are in shared memory
// anyway).  Measured against contiguous runs of one row tile per CTA, whose
// 64 concurrent row tiles (128 MB of A at 16384 × 4096) overflow L2: 353 ->
// 336 us at M, K, N = 16384, 4096, 4096 and 1600 -> 1346 us at 32768, 4096,
// 8192, with bitwise equal results.
constexpr int kGroup2 = 8;
constexpr int kBM2 = 2 * kBM;
constexpr int kBoxA2 = kBM2 * kBK * 2;           // 32 KB
constexpr int kBoxB2 = 256 * kBK * 2;            // 32 KB
constexpr int kStage2 = kBoxA2 + kBoxB2;         // 64 KB
constexpr int kStages2 = 3;
constexpr int kSs2Bytes = 2 * kBM2 * 4;          // square sums, double-buffered
constexpr int kBar2Bytes = 256;
constexpr int kSmem2 = 1024 + kStages2 * kStage2 + kSs2Bytes + kBar2Bytes;
static_assert(kSmem2 <= 227 * 1024, "shared memory");

// The whole 256 × 256 tiles of a CTA: tile indices t = cta, cta + grid, ...
// below `end`, each mapped to (row tile, column tile) by the grouped order.
struct TIter {
    int64_t t, end;
    int n_tiles, stride, m_tiles;
    __device__ bool next(Segment &s) {
        if (t >= end) return false;
        const int64_t per_group = static_cast<int64_t>(kGroup2) * n_tiles;
        const int g = static_cast<int>(t / per_group);
        const int w = static_cast<int>(t - static_cast<int64_t>(g) * per_group);
        const int left = m_tiles - g * kGroup2;  // row tiles in this group
        const int rows = left < kGroup2 ? left : kGroup2;
        s.m = g * kGroup2 + w % rows;
        s.n = w / rows;
        s.k0 = 0;
        s.k1 = 0;  // unused: every tile runs all K blocks
        t += stride;
        return true;
    }
};

struct M2Bars {
    uint64_t *full, *empty;   // [kStages2]
    uint64_t *acc_full;       // MMA -> epilogue, one phase per tile
    uint64_t *acc_empty;      // [2] epilogue -> MMA, per accumulator
    uint64_t *ss_full, *ss_empty;  // [2]
    uint64_t *drain;
    uint32_t *tmem_holder;
};

__device__ void m2_producer(const pipe::Pipe &p, const M2Bars &b, TIter it, int kbt,
                            const CUtensorMap *tm_a, const CUtensorMap *tm_b)
{
    const uint64_t pol_a = ptx::policy_evict_normal();  // read by the group's other column tiles
    const uint64_t pol_b = ptx::policy_evict_last();    // re-read by every row tile
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0, issued_parity = 0;
    Segment sg;
    bool ok = true;
    while (ok && it.next(sg)) {
        for (int kb = 0; kb < kbt; ++kb) {
            if (!pipe::wait(p, &b.empty[stage], phase ^ 1)) {
                ok = false;
                break;
            }
            uint8_t *a = p.stages + stage * kStage2;
            ptx::mbar_arrive_expect_tx(&b.full[stage], kStage2);
            ptx::tma_load_2d(a, tm_a, kb * kBK, sg.m * kBM2, &b.full[stage], pol_a);
            ptx::tma_load_2d(a + kBoxA2, tm_b, kb * kBK, sg.n * 256, &b.full[stage], pol_b);
            issued_mask |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            if (++stage == kStages2) { stage = 0; phase ^= 1; }
        }
    }
    if (!ok) {
        for (int s = 0; s < kStages2; ++s) {
            if (!((issued_mask >> s) & 1u)) continue;
            volatile int never = 0;
            ptx::mbar_wait_bounded(&b.full[s], (issued_parity >> s) & 1u, &never, p.limit_ns);
        }
    }
}

__device__ void m2_mma_issuer(const pipe::Pipe &p, const M2Bars &b, TIter it, int kbt)
{
    constexpr uint32_t idesc = ptx::idesc_bf16_f32(kBM, 256);
    int stage = 0;
    uint32_t phase = 0;
    int seg = 0;
    Segment sg;
    bool ok = true;
    while (ok && it.next(sg)) {
        const uint32_t epar = (seg & 1) ^ 1;  // each accumulator freed from the previous tile
        for (int kb = 0; kb < kbt && ok; ++kb) {
            if (!pipe::wait(p, &b.full[stage], phase)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t a_addr = ptx::smem_u32(p.stages + stage * kStage2);
            const uint64_t b_desc = ptx::smem_desc_sw128(a_addr + kBoxA2);
            for (int h = 0; h < 2; ++h) {
                if (kb == 0) {
                    if (!pipe::wait(p, &b.acc_empty[h], epar)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                }
                // rows 128·h.. of the A box: 16 KB on, the same 128-byte swizzle
                const uint64_t a_desc = ptx::smem_desc_sw128(a_addr + h * (kBoxA2 / 2));
                const uint32_t d_tmem = p.tmem_base + static_cast<uint32_t>(h * 256);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    ptx::mma_bf16(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, idesc,
                                  (kb > 0 || kk > 0) ? 1u : 0u);
            }
            if (!ok) break;
            ptx::mma_commit(&b.empty[stage]);
            if (++stage == kStages2) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        ptx::mma_commit(b.acc_full);
        ++seg;
    }
    if (!ok || *p.abort) {
        ptx::mma_commit(b.drain);
        volatile int never = 0;
        ptx::mbar_wait_bounded(b.drain, 0, &never, p.limit_ns);
    }
}


// Thread t sums rows t and t + 128 of the tile; a tile of the previous tile's
// row tile (rare in the grouped order) reuses its sums.
__device__ void m2_square_sums(const pipe::Pipe &p, const M2Bars &b, TIter it, int kbt, int t,
                               int lane)
{
    int stage = 0;
    uint32_t phase = 0;
    int seg = 0;
    int prev_m = -1;
    float prev0 = 0.f, prev1 = 0.f;
    Segment sg;
    bool ok = true;
    while (ok && it.next(sg)) {
        const bool reuse = sg.m == prev_m;
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
        for (int kb = 0; kb < kbt; ++kb) {
            if (!pipe::wait(p, &b.full[stage], phase)) {
                ok = false;
                break;
            }
            if (!reuse) {
                const uint8_t *base = p.stages + stage * kStage2;
                row_sq64(base + t * 128, t, s0);
                row_sq64(base + (t + kBM) * 128, t + kBM, s1);
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&b.empty[stage]);
            if (++stage == kStages2) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        const float ss0 = reuse ? prev0 : (s0[0] + s0[1]) + (s0[2] + s0[3]);
        const float ss1 = reuse ? prev1 : (s1[0] + s1[1]) + (s1[2] + s1[3]);
        const int buf = seg & 1;
        if (!pipe::wait(p, &b.ss_empty[buf], ((seg >> 1) & 1) ^ 1)) break;
        p.ss_buf[buf * kBM2 + t] = ss0;
        p.ss_buf[buf * kBM2 + kBM + t] = ss1;
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&b.ss_full[buf]);
        prev_m = sg.m;
        prev0 = ss0;
        prev1 = ss1;
        ++seg;
    }
}

__global__ void __launch_bounds__(kThreads, 1)
rmsnorm_gemm_m256_kernel(const __grid_constant__ CUtensorMap tm_a,
                         const __grid_constant__ CUtensorMap tm_b, int64_t M, int64_t N, int K,
                         float eps, int64_t tiles, int n_tiles, uint16_t *__restrict__ Cout,
                         uint64_t wait_limit_ns)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    pipe::Pipe p{};
    p.stages = smem;
    p.ss_buf = reinterpret_cast<float *>(smem + kStages2 * kStage2);  // [2][256]
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kStages2 * kStage2 + kSs2Bytes);
    M2Bars b;
    b.full = bar;
    b.empty = bar + kStages2;
    b.acc_full = bar + 2 * kStages2;
    b.acc_empty = b.acc_full + 1;
    b.ss_full = b.acc_empty + 2;
    b.ss_empty = b.ss_full + 2;
    b.drain = b.ss_empty + 2;
    b.tmem_holder = reinterpret_cast<uint32_t *>(b.drain + 1);
    p.abort = reinterpret_cast<volatile int *>(b.tmem_holder + 1);
    p.status = &g_rng_status;
    p.limit_ns = wait_limit_ns;
    p.stages_n = kStages2;
    p.stage_bytes = kStage2;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const int kbt = (K + kBK - 1) / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages2; ++s) {
            ptx::mbar_init(&b.full[s], 1);
            ptx::mbar_init(&b.empty[s], 1 + 4);  // MMA commit + one arrive per square-sum warp
        }
        ptx::mbar_init(b.acc_full, 1);
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&b.acc_empty[a], 4);
            ptx::mbar_init(&b.ss_full[a], 4);
            ptx::mbar_init(&b.ss_empty[a], 4);
        }
        ptx::mbar_init(b.drain, 1);
        *p.abort = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tm_a);
        ptx::prefetch_tensormap(&tm_b);
    }
    if (warp == 1) ptx::tmem_alloc<512>(b.tmem_holder);
    ptx::tc_fence_before();
    __syncwarp();
    __syncthreads();
    ptx::tc_fence_after();
    p.tmem_base = *b.tmem_holder;
    ptx::pdl_wait();

    const TIter segs{cta, tiles, n_tiles, static_cast<int>(gridDim.x),
                     static_cast<int>(tiles / n_tiles)};
    const float inv_k = 1.0f / static_cast<float>(K);

    if (warp == 0) {
        if (lane == 0) m2_producer(p, b, segs, kbt, &tm_a, &tm_b);
    } else if (warp == 1) {
        if (lane == 0) m2_mma_issuer(p, b, segs, kbt);
    } else if (warp < 6) {
        m2_square_sums(p, b, segs, kbt, (warp - 2) * 32 + lane, lane);
    } else {
        // ----------------------------------------------- epilogue (warps 6..9)
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        int seg = 0;
        TIter it = segs;
        Segment sg;
        while (it.next(sg)) {
            if (!pipe::wait(p, b.acc_full, seg & 1)) break;
            ptx::tc_fence_after();
            const int buf = seg & 1;
            if (!pipe::wait(p, &b.ss_full[buf], (seg >> 1) & 1)) break;
            const float ss0 = p.ss_buf[buf * kBM2 + row];
            const float ss1 = p.ss_buf[buf * kBM2 + kBM + row];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&b.ss_empty[buf]);
            ++seg;
            const int64_t col0 = static_cast<int64_t>(sg.n) * 256;
            for (int h = 0; h < 2; ++h) {
                const int64_t grow = static_cast<int64_t>(sg.m) * kBM2 + h * kBM + row;
                const float rstd = rsqrtf((h ? ss1 : ss0) * inv_k + eps);
                const uint32_t taddr = p.tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                       static_cast<uint32_t>(h * 256);
#pragma unroll 1
                for (int j = 0; j < 8; ++j) {
                    float v[32], t16[16];
                    ptx::tmem_ld_16(taddr + j * 32, t16);
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = t16[e];
                    ptx::tmem_ld_16(taddr + j * 32 + 16, t16);
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[16 + e] = t16[e];
                    ptx::tmem_ld_wait();
                    const int64_t c0 = col0 + j * 32;
                    if (grow < M && c0 < N) {
                        const int valid = N - c0 < 32 ? static_cast<int>(N - c0) : 32;
                        if (in_range(708, grow, 1, M) && in_range(709, c0, (valid + 7) / 8 * 8, N))
                            store_cols32(v, rstd, Cout + grow * N + c0, valid);
                    }
                    __syncwarp();  // the next tcgen05.ld is warp-collective
                }
                // this accumulator may take the next tile's first MMAs
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&b.acc_empty[h]);
            }
        }
    }

    // lane 0 of the TMA and MMA warps ran alone: reconverge every warp before
    // the CTA barrier, which needs whole warps
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::pdl_trigger();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc<512>(p.tmem_base);
    }
}

__global__ void zero_ints_kernel(int *p, int64_t count)
{
    ptx::pdl_wait();
    ptx::pdl_trigger();
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        p[i] = 0;
}

int tile_cols(int64_t N) { return N <= 32 ? 32 : (N <= 64 ? 64 : (N <= 128 ? 128 : 256)); }

RSched rng_sched(int64_t M, int64_t K, int64_t N, int num_sms)
{
    const int NT = tile_cols(N);
    RSched s{};
    s.n_tiles = static_cast<int>((N + NT - 1) / NT);
    s.tiles = (M + kBM - 1) / kBM * s.n_tiles;
    s.kbt = static_cast<int>((K + kBK - 1) / kBK);
    s.total = s.tiles * s.kbt;
    if (s.tiles >= num_sms) {  // whole tiles only
        s.aligned = 1;
        s.grid = num_sms;
    } else {  // K split over the CTAs of a tile
        s.aligned = 0;
        int64_t g = num_sms;
        if (g > kMaxFanIn * s.tiles) g = kMaxFanIn * s.tiles;
        if (g > s.total) g = s.total;
        s.grid = static_cast<int>(g < 1 ? 1 : g);
    }
    return s;
}

size_t tickets_bytes(int64_t tiles) { return (static_cast<size_t>(tiles) * 4 + 255) / 256 * 256; }

// 256 × 256 tiles when every SM gets at least one and K has at least 64
// blocks.  Their accumulators are single-buffered, so a tile's epilogue holds
// up the next tile's first MMAs for a few µs; below 64 K blocks that costs more
// than the smaller stages gain.
bool m256_ok(int64_t M, int64_t K, int64_t N, int num_sms)
{
    return tile_cols(N) == 256 && (K + kBK - 1) / kBK >= 64 &&
           (M + kBM2 - 1) / kBM2 * ((N + 255) / 256) >= num_sms;
}

cudaError_t launch_m256(const uint16_t *A, const uint16_t *B_t, int64_t M, int64_t K, int64_t N,
                        float eps, uint16_t *C, int num_sms, int device, cudaStream_t stream)
{
    CUtensorMap ta, tb;
    if (!make_tmap(&ta, A, static_cast<uint64_t>(K), static_cast<uint64_t>(M), kBM2) ||
        !make_tmap(&tb, B_t, static_cast<uint64_t>(K), static_cast<uint64_t>(N), 256))
        return cudaErrorInvalidValue;
    static uint64_t configured = 0;  // one bit per device
    static std::mutex mu;
    if (device < 64 && !((configured >> device) & 1)) {
        std::lock_guard<std::mutex> lock(mu);
        cudaError_t e = cudaFuncSetAttribute(rmsnorm_gemm_m256_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem2);
        if (e != cudaSuccess) return e;
        configured |= 1ull << device;
    }
    const int64_t tiles = (M + kBM2 - 1) / kBM2 * ((N + 255) / 256);
    return launch_pdl(rmsnorm_gemm_m256_kernel, dim3(num_sms), dim3(kThreads), kSmem2, stream,
                      ta, tb, M, N, static_cast<int>(K), eps, tiles,
                      static_cast<int>((N + 255) / 256), C, kWaitLimitNs);
}

template <int NT>
cudaError_t launch_nt(const CUtensorMap &ta, const CUtensorMap &tb, int64_t M, int64_t N, int K,
                      float eps, const RSched &s, uint16_t *C, int *tickets, float *partials,
                      int device, uint64_t limit, cudaStream_t stream)
{
    using R = RCfg<NT>;
    static uint64_t configured = 0;  // one bit per device
    static std::mutex mu;
    if (device < 64 && !((configured >> device) & 1)) {
        std::lock_guard<std::mutex> lock(mu);
        cudaError_t e = cudaFuncSetAttribute(rmsnorm_gemm_kernel<NT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             R::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured |= 1ull << device;
    }
    return launch_pdl(rmsnorm_gemm_kernel<NT>, dim3(s.grid), dim3(kThreads), R::kSmemBytes,
                      stream, ta, tb, M, N, K, eps, s, C, tickets, partials, limit);
}

}  // namespace

size_t rmsnorm_gemm_workspace_bytes(int64_t M, int64_t K, int64_t N, int num_sms)
{
    if (M <= 0) return 0;
    if (m256_ok(M, K, N, num_sms)) return 0;
    const RSched s = rng_sched(M, K, N, num_sms);
    if (s.aligned) return 0;
    const size_t slots = static_cast<size_t>(s.grid) + static_cast<size_t>(s.tiles);
    return tickets_bytes(s.tiles) + slots * kBM * (tile_cols(N) + 1) * sizeof(float);
}

cudaError_t launch_rmsnorm_gemm(const uint16_t *A, const uint16_t *B_t, int64_t M, int64_t K,
                                int64_t N, float eps, uint16_t *C, void *workspace, int num_sms,
                                cudaStream_t stream)
{
    int device = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&device)) != cudaSuccess) return e;
    if (m256_ok(M, K, N, num_sms)) return launch_m256(A, B_t, M, K, N, eps, C, num_sms, device, stream);
    const RSched s = rng_sched(M, K, N, num_sms);
    const int NT = tile_cols(N);
    CUtensorMap ta, tb;
    if (!make_tmap(&ta, A, static_cast<uint64_t>(K), static_cast<uint64_t>(M), kBM) ||
        !make_tmap(&tb, B_t, static_cast<uint64_t>(K), static_cast<uint64_t>(N),
                   static_cast<uint32_t>(NT)))
        return cudaErrorInvalidValue;
    int *tickets = nullptr;
    float *partials = nullptr;
    if (!s.aligned) {
        tickets = static_cast<int *>(workspace);
        partials = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                             tickets_bytes(s.tiles));
        const int64_t blocks = (s.tiles + 255) / 256 < 64 ? (s.tiles + 255) / 256 : 64;
        e = launch_pdl(zero_ints_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                       tickets, s.tiles);
        if (e != cudaSuccess) return e;
    }
    const int Ki = static_cast<int>(K);
    switch (NT) {
    case 32: return launch_nt<32>(ta, tb, M, N, Ki, eps, s, C, tickets, partials, device, kWaitLimitNs, stream);
    case 64: return launch_nt<64>(ta, tb, M, N, Ki, eps, s, C, tickets, partials, device, kWaitLimitNs, stream);
    case 128: return launch_nt<128>(ta, tb, M, N, Ki, eps, s, C, tickets, partials, device, kWaitLimitNs, stream);
    default: return launch_nt<256>(ta, tb, M, N, Ki, eps, s, C, tickets, partials, device, kWaitLimitNs, stream);
    }
}

cudaError_t read_and_clear_rmsnorm_gemm_status(int *status)
{
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    int v = 0, zero = 0;
    if ((e = cudaMemcpyFromSymbol(&v, g_rng_status, sizeof v)) != cudaSuccess) return e;
    if ((e = cudaMemcpyToSymbol(g_rng_status, &zero, sizeof zero)) != cudaSuccess) return e;
    *status = v;
    return cudaSuccess;
}

}  // namespace mhc
