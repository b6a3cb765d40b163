// Steps 1–4a of the mHC forward in one persistent kernel, reading X from HBM
// once for both the projection GEMM and the pre-mixing (page "mHC 算法分析 &
// cutile 高效实现", §2.1–§2.5; the page's advice not to let intermediates land
// in memory, §3.4, applied across the GEMM and the pre-apply):
//
//   Y = X·φ, r = sqrt(Σx²/K)                 (S1)
//   H_pre, H_post, H_res = coefficients(Y,r)  (S2, S3)
//   F_pre = Σ_i H_pre[i]·X[i]                 (S4a)
//
// The batch is walked in chunks of CH token tiles (128 tokens each).  Every
// CTA works on every chunk: the G = CH·P CTAs are P "contributors" per tile,
// and contributor p of a tile takes K blocks [kbt·p/P, kbt·(p+1)/P) of it
// through the TMA → tcgen05 pipeline of gemm_pipeline.cuh (X loaded with the
// evict_normal L2 policy), parks its partial row sums in global memory and
// later finishes its own rows [128·p/P, 128·(p+1)/P) of the tile: the fixed-
// order sum of the P partials, Y and r, the coefficients, and F_pre from a
// second read of those rows' X.  That read hits L2 because the producer is
// held back (LeadIter) until at most `lead` chunks of X have been streamed
// and not yet re-read.  Sixteen warps per CTA:
//   warps 0-5   the pipeline: TMA (throttled), MMA, square-sum;
//   warps 6-9   epilogue: park this CTA's partial of each tile (row sums of Y
//               and Σx²), count it in the tile's ticket, then finish the rows
//               of the tile before (whose partials have had a segment's time
//               to arrive): the fixed-order sum of its P partials, all loads
//               issued at once, then Y and r;
//   warps 10-13 finisher: H_pre of the finished rows (σ only), then F_pre of
//               each piece from shared memory;
//   warp 14     coefficients: H_pre, H_post and the Sinkhorn–Knopp H_res of
//               the rows (token_coeffs, as the standalone kernel);
//   warp 15     loader: once the tile's P partials are in (its X has just
//               streamed through L2), bulk-copies the CTA's rows of X, piece
//               by piece, into a ring of shared-memory slots.
// Partials rotate through nb buffers by chunk; before reusing one a CTA waits
// (bounded) until the P finishers of that buffer's previous tile have read it.
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

constexpr int kThreads = 512;   // 16 warps (see above)
constexpr int kEpiT = 128;
constexpr int kPreT = 128;
constexpr int kMaxRows = 16;    // rows each contributor finishes per tile (P >= 8)
constexpr int kRowBufs = 4;     // finished-row buffers in flight
constexpr int kSlotBytes = 8192;  // one piece of the X re-read
constexpr int kReduceBatch = 40;  // partials in flight per thread of the fixed-order sums
// X bytes per chunk and chunks streamed ahead of the re-read (see LeadIter,
// >= 2).  Measured at B=16384, n=4, C=7168: 4-tile chunks (29 MB) with lead 3
// were fastest, though about a third of the re-read then misses L2; 2-tile
// chunks keep it in L2 but pay the per-tile latencies twice as often.
constexpr int64_t kChunkBytes = 32LL << 20;
constexpr int kLeadChunks = 3;
constexpr int kMaxPartBufs = 8;
static_assert(kLeadChunks >= 2, "see LeadIter");

__device__ int g_fused_status;

template <int n>
struct FCfg {
    static constexpr int N = n * n + 2 * n;
    static constexpr int NPAD = (N + 15) / 16 * 16;
    // n <= 4: a 4-stage GEMM ring and 15 re-read slots.  The producer is held
    // back by LeadIter anyway, and the re-read is the latency-bound side:
    // measured at B=16384, C=7168, 6 stages and 10 slots took 663.5 us per
    // forward, 5 and 12 took 660.1, 4 and 15 took 656.6 (at B=4096, C=4096:
    // 107.2, 106.6, 106.2 us).
    static constexpr int kRingBudget = n <= 4 ? 84 * 1024 : 134 * 1024;
    static constexpr int kSlots = n <= 4 ? 15 : 8;  // X re-read slots (shared memory left over)
    // n <= 4: the epilogue stages its partial in shared memory and stores it
    // coalesced; wider rows do not fit and are stored from registers
    static constexpr bool kStage = n <= 4;
    static constexpr int kStageBytes = kStage ? kBM * (N + 1) * 4 : 0;
    using C = pipe::Cfg<NPAD, kRingBudget>;
    // channels per piece: one pass of the 128 pre-apply threads (8 each), n streams per slot
    static constexpr int kW = (kSlotBytes / (2 * n)) / 8 * 8 < 8 * kPreT
                                  ? (kSlotBytes / (2 * n)) / 8 * 8
                                  : 8 * kPreT;
    static constexpr int kRowsBytes = kRowBufs * kMaxRows * (N + 1) * 4;
    static constexpr int kHpBytes = kMaxRows * 8 * 4;
    static constexpr int kRedBytes = kPreT * 4;                      // group sums of the reduction
    static constexpr int kOwnBarBytes = 384;                         // barriers of this kernel
    static constexpr int kSmemBytes = 1024 + C::kRingBytes + pipe::kSsBytes + pipe::kBarrierBytes +
                                      kSlots * kSlotBytes + kRowsBytes + kHpBytes + kRedBytes +
                                      kStageBytes + kOwnBarBytes;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
    static_assert(kW % 8 == 0 && kW / 8 <= kPreT, "a piece is one pass of the pre-apply warps");
    static_assert((2 + 2 * kRowBufs + 2 * kSlots) * 8 + 4 <= kOwnBarBytes, "barrier area");
    static_assert(!kStage || (32 * (N + 1)) % 4 == 0, "a warp's staged rows are whole float4s");
};

struct FSched {
    int m_tiles, kbt, CH, P, nchunks;
    int lead;  // chunks the GEMM may run ahead of this CTA's finished pre-apply
    int nb;    // partial buffers, used in turn by consecutive chunks
};

// The segments of the CTA in tile slot j, contributor p: one per chunk.
struct ChunkIter {
    FSched s;
    int j, p, c;
    __device__ bool next(Segment &sg) {
        while (c < s.nchunks) {
            const int t = c * s.CH + j;
            ++c;
            if (t >= s.m_tiles) continue;  // the last chunk may hold fewer tiles
            sg.m = t;
            sg.k0 = s.kbt * p / s.P;
            sg.k1 = s.kbt * (p + 1) / s.P;
            return true;
        }
        return false;
    }
};

// The producer's segments, each released only once the pre-apply warps of
// this CTA have finished the segment `lead` places back: the X streamed for
// the GEMM but not yet re-read stays within `lead` chunks, which is what has
// to fit in L2.  lead >= 2: the epilogue finishes a tile's rows after parking
// the next tile, so with lead = 1 a segment would wait for its own park.  On a
// timeout or an abort the segment is still returned; the producer's next
// stage wait then sees the abort and drains its copies.
struct LeadIter {
    ChunkIter it;
    const volatile int *pre_done;  // segments the pre-apply warps have finished
    const pipe::Pipe *p;
    int seg;
    __device__ bool next(Segment &sg) {
        if (!it.next(sg)) return false;
        const int need = seg + 1 - it.s.lead;
        ++seg;
        if (need <= 0) return true;
        const uint64_t t0 = ptx::globaltimer_ns();
        for (uint32_t polls = 0; *pre_done < need; ++polls) {
            if ((polls & 63) == 63) {
                if (*p->abort) return true;
                if (ptx::globaltimer_ns() - t0 > p->limit_ns) {
                    pipe::raise_timeout(*p);
                    return true;
                }
            }
            __nanosleep(32);
        }
        return true;
    }
};

// Bounded wait until the global counter reaches `target` (acquire).
__device__ bool wait_count(const pipe::Pipe &p, const int *addr, int target)
{
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t polls = 0;; ++polls) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
        if (v >= target) return true;
        if ((polls & 31) == 31) {
            if (*p.abort) return false;
            if (polls >= 4096 && ptx::globaltimer_ns() - t0 > p.limit_ns) {
                pipe::raise_timeout(p);
                return false;
            }
        }
        __nanosleep(64);
    }
}

__device__ __forceinline__ int clamp_rows(int r0, int r1, int valid)
{
    const int hi = r1 < valid ? r1 : valid;
    return hi > r0 ? hi - r0 : 0;
}

// Σ over contributors q in [q0, q1) of src[q·qs], in order, kReduceBatch loads
// in flight at a time (s + 0 is exact for the padding).
__device__ __forceinline__ float partial_sum(const float *src, int64_t qs, int q0, int q1)
{
    float s = 0.f;
    for (int q = q0; q < q1; q += kReduceBatch) {
        float vb[kReduceBatch];
#pragma unroll
        for (int u = 0; u < kReduceBatch; ++u)
            vb[u] = q + u < q1 ? __ldcg(src + static_cast<int64_t>(q + u) * qs) : 0.f;
#pragma unroll
        for (int u = 0; u < kReduceBatch; ++u) s += vb[u];
    }
    return s;
}

template <int n>
__global__ void __launch_bounds__(kThreads, 1)
fused_pre_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                 int64_t B, int K, int C, FSched fs, float a_pre, float a_post, float a_res,
                 const float *__restrict__ bias, int iters, const uint16_t *X,
                 float *__restrict__ Y, float *__restrict__ r, float *__restrict__ H_pre,
                 float *__restrict__ H_post, float *__restrict__ H_res,
                 uint16_t *__restrict__ F_pre, int *tickets, int *done, float *partials,
                 uint64_t wait_limit_ns)
{
    using F = FCfg<n>;
    constexpr int N = F::N;
    constexpr int NPAD = F::NPAD;
    constexpr int stride = N + 1;  // a finished row: N sums of Y, then r
    constexpr int W = F::kW;
    constexpr int kSlots = F::kSlots;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    pipe::Pipe p;
    uint8_t *after = pipe::carve<NPAD, F::kRingBudget>(p, smem, &g_fused_status, wait_limit_ns);
    uint8_t *slots = after;                                             // [kSlots][kSlotBytes]
    float *rows_buf = reinterpret_cast<float *>(slots + kSlots * kSlotBytes);  // [kRowBufs][kMaxRows][stride]
    float *hp_buf = rows_buf + kRowBufs * kMaxRows * stride;            // [kMaxRows][8]
    float *red = hp_buf + kMaxRows * 8;                                 // [kEpiT]
    float *stage = red + kEpiT;                                         // [kBM][stride] if F::kStage
    uint64_t *epi_bar = reinterpret_cast<uint64_t *>(stage + F::kStageBytes / 4);
    uint64_t *pre_bar = epi_bar + 1;
    uint64_t *rows_full = pre_bar + 1;            // [kRowBufs] epilogue -> finisher, coefficients
    uint64_t *rows_empty = rows_full + kRowBufs;  // [kRowBufs] finisher, coefficients -> epilogue
    uint64_t *slot_full = rows_empty + kRowBufs;  // [kSlots] loader -> finisher
    uint64_t *slot_empty = slot_full + kSlots;    // [kSlots] finisher -> loader
    volatile int *pre_done = reinterpret_cast<volatile int *>(slot_empty + kSlots);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = blockIdx.x;
    const int j = g / fs.P, pc = g - (g / fs.P) * fs.P;  // tile slot, contributor
    const int G = fs.CH * fs.P;
    const int r0 = kBM * pc / fs.P, r1 = kBM * (pc + 1) / fs.P;  // rows this CTA finishes
    // one CTA's partial: [kBM][N + 1] (N sums of Y, then Σx²); nb·G of them
    const int64_t part_stride = static_cast<int64_t>(kBM) * stride;
    const int64_t part_slots = static_cast<int64_t>(fs.nb) * G;

    if (threadIdx.x == 0) {
        pipe::init_barriers(p);
        ptx::mbar_init(epi_bar, kEpiT);
        ptx::mbar_init(pre_bar, kPreT);
        for (int a = 0; a < kRowBufs; ++a) {
            ptx::mbar_init(&rows_full[a], 1);
            ptx::mbar_init(&rows_empty[a], 2);  // finisher + coefficient warp
        }
        for (int a = 0; a < kSlots; ++a) {
            ptx::mbar_init(&slot_full[a], 1);
            ptx::mbar_init(&slot_empty[a], 4);
        }
        *pre_done = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tm_x);
        ptx::prefetch_tensormap(&tm_w);
    }
    if (warp == 1) ptx::tmem_alloc<F::C::kTmemCols>(p.tmem_holder);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    p.tmem_base = *p.tmem_holder;
    ptx::pdl_wait();  // global memory only after the previous kernel has completed

    const ChunkIter segs{fs, j, pc, 0};

    if (warp == 0) {
        if (lane == 0)  // X stays in L2 until the loader re-reads it
            pipe::producer<NPAD>(p, LeadIter{segs, pre_done, &p, 0}, &tm_x, &tm_w,
                                 ptx::policy_evict_normal(), -1);
    } else if (warp == 1) {
        if (lane == 0) pipe::mma_issuer<NPAD>(p, segs);
    } else if (warp < 6) {
        pipe::square_sum<NPAD>(p, segs, (warp - 2) * 32 + lane, lane);
    } else if (warp < 10) {
        // ------------------------------------------ epilogue (warps 6..9)
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        const int et = threadIdx.x - 192;
        uint32_t epi_phase = 0;

        // Finishes rows [r0, r0 + nrows) of the tile of segment fseg: item
        // e = row·stride + column, summed over the P partials in contributor
        // order (with few items the contributors are split into `groups`
        // ranges whose sums are added in range order); then Y, r and the row
        // buffer for the finisher and the coefficient warp.
        auto finish = [&](int fseg, int t) -> bool {
            const int c = t / fs.CH;
            const int64_t row0 = static_cast<int64_t>(t) * kBM;
            const int valid = static_cast<int>(B - row0 < kBM ? B - row0 : kBM);
            const int nrows = clamp_rows(r0, r1, valid);
            const int rb = fseg % kRowBufs;
            float *rows = rows_buf + rb * kMaxRows * stride;
            if (!pipe::wait(p, &rows_empty[rb], ((fseg / kRowBufs) & 1) ^ 1)) return false;
            if (!in_range(501, t, 1, fs.m_tiles) ||
                !in_range(502, static_cast<int64_t>(c % fs.nb) * G + static_cast<int64_t>(j) * fs.P,
                          fs.P, part_slots) ||
                !in_range(503, row0 + r0, nrows, B))
                return false;
            if (et == 0) wait_count(p, &tickets[t], fs.P);
            // the acquire above and the group barrier order the partial loads
            if (!pipe::group_sync(p, epi_bar, epi_phase) || *p.abort) return false;
            const int E = nrows * stride;
            const float *base =
                partials + (static_cast<int64_t>(c % fs.nb) * G + static_cast<int64_t>(j) * fs.P) *
                               part_stride + static_cast<int64_t>(r0) * stride;
            auto emit = [&](int e, float s) {
                const int rr = e / stride, cc = e - (e / stride) * stride;
                const float out = cc < N ? s : sqrtf(s / static_cast<float>(K));
                if (cc < N)
                    Y[(row0 + r0 + rr) * N + cc] = out;
                else
                    r[row0 + r0 + rr] = out;
                rows[rr * stride + cc] = out;
            };
            const int groups = E >= kEpiT || E == 0 ? 1 : kEpiT / E;
            if (groups == 1) {
                for (int e = et; e < E; e += kEpiT) emit(e, partial_sum(base + e, part_stride, 0, fs.P));
            } else {
                const int gi = et / E, e = et - (et / E) * E;
                if (gi < groups)
                    red[gi * E + e] = partial_sum(base + e, part_stride, fs.P * gi / groups,
                                                  fs.P * (gi + 1) / groups);
                if (!pipe::group_sync(p, epi_bar, epi_phase)) return false;
                if (et < E) {
                    float s = red[et];
                    for (int g2 = 1; g2 < groups; ++g2) s += red[g2 * E + et];
                    emit(et, s);
                }
            }
            if (!pipe::group_sync(p, epi_bar, epi_phase)) return false;
            if (et == 0) {
                atomicAdd(&done[t], 1);  // this CTA has read the tile's partials
                ptx::mbar_arrive(&rows_full[rb]);
            }
            return true;
        };

        // Park each tile's partial, then finish the previous tile, whose
        // partials have had a segment's time to arrive.
        int seg = 0, prev_t = -1;
        bool ok = true;
        ChunkIter it = segs;
        Segment sg;
        while (it.next(sg)) {
            float v[NPAD];
            float ss;
            if (!pipe::take_accumulator<NPAD>(p, seg, q, lane, v, ss)) {
                ok = false;
                break;
            }
            const int t = sg.m;
            const int c = t / fs.CH;
            const int64_t row0 = static_cast<int64_t>(t) * kBM;
            const int valid = static_cast<int>(B - row0 < kBM ? B - row0 : kBM);

            if (!in_range(504, t, 1, fs.m_tiles) ||
                !in_range(505, static_cast<int64_t>(c % fs.nb) * G + g, 1, part_slots)) {
                ok = false;
                break;
            }
            // this buffer was last used for tile t - nb·CH: wait for its P readers
            if (c >= fs.nb && et == 0) wait_count(p, &done[t - fs.nb * fs.CH], fs.P);
            if (!pipe::group_sync(p, epi_bar, epi_phase) || *p.abort) {
                ok = false;
                break;
            }
            float *mine = partials + (static_cast<int64_t>(c % fs.nb) * G + g) * part_stride;
            if constexpr (F::kStage) {
                // this warp's 32 rows through shared memory, then 16-byte stores
                // of the contiguous block (rows past the batch hold zeros and
                // are never read)
                float *st = stage + q * 32 * stride;
#pragma unroll
                for (int k = 0; k < NPAD; ++k)
                    if (k < N) st[lane * stride + k] = v[k];
                st[lane * stride + N] = ss;
                __syncwarp();
                const float4 *src4 = reinterpret_cast<const float4 *>(st);
                float4 *dst4 = reinterpret_cast<float4 *>(mine + q * 32 * stride);
                for (int f = lane; f < 32 * stride / 4; f += 32) __stcg(dst4 + f, src4[f]);
                __syncwarp();
            } else if (row < valid) {
#pragma unroll
                for (int k = 0; k < NPAD; ++k)
                    if (k < N) mine[row * stride + k] = v[k];
                mine[row * stride + N] = ss;
            }
            if (!pipe::group_sync(p, epi_bar, epi_phase)) {
                ok = false;
                break;
            }
            if (et == 0) {  // release: the group's stores, then the ticket
                __threadfence();
                atomicAdd(&tickets[t], 1);
            }
            if (seg > 0 && !finish(seg - 1, prev_t)) {
                ok = false;
                break;
            }
            prev_t = t;
            ++seg;
        }
        if (ok && seg > 0) finish(seg - 1, prev_t);
    } else if (warp < 14) {
        // ----------------------------------------- finisher (warps 10..13)
        const int pt = threadIdx.x - 320;
        uint32_t pre_phase = 0;
        int slot = 0;
        uint32_t slot_phase = 0;
        int seg = 0;
        ChunkIter it = segs;
        Segment sg;
        bool ok = true;
        while (ok && it.next(sg)) {
            const int t = sg.m;
            const int64_t row0 = static_cast<int64_t>(t) * kBM;
            const int valid = static_cast<int>(B - row0 < kBM ? B - row0 : kBM);
            const int nrows = clamp_rows(r0, r1, valid);
            const int rb = seg % kRowBufs;
            if (!pipe::wait(p, &rows_full[rb], (seg / kRowBufs) & 1)) break;
            // H_pre of the finished rows (σ only; the coefficient warp writes it)
            if (pt < nrows * n) {
                const int tk = pt / n, i = pt - (pt / n) * n;
                const float *yrow = rows_buf + (rb * kMaxRows + tk) * stride;
                hp_buf[tk * 8 + i] = pre_coeff(yrow[i], 1.0f / yrow[N], a_pre, bias[i]);
            }
            if (!pipe::group_sync(p, pre_bar, pre_phase)) break;
            if (pt == 0) ptx::mbar_arrive(&rows_empty[rb]);
            // F_pre of each piece, in the loader's order
            for (int tk = 0; tk < nrows && ok; ++tk) {
                float h[n];
#pragma unroll
                for (int k = 0; k < n; ++k) h[k] = hp_buf[tk * 8 + k];
                const int64_t tok = row0 + r0 + tk;
                const bool tok_ok = in_range(506, tok, 1, B);
                for (int c0 = 0; c0 < C; c0 += W) {
                    const int wp = C - c0 < W ? C - c0 : W;
                    if (!pipe::wait(p, &slot_full[slot], slot_phase)) {
                        ok = false;
                        break;
                    }
                    if (pt * 8 < wp && tok_ok && in_range(507, c0 + pt * 8, 8, C)) {
                        const uint8_t *sl = slots + slot * kSlotBytes;
                        uint4 xv[n];
#pragma unroll
                        for (int k = 0; k < n; ++k)
                            xv[k] = *reinterpret_cast<const uint4 *>(sl + k * wp * 2 + pt * 16);
                        ptx::st_stream_v4(F_pre + tok * C + c0 + pt * 8, pre_mix8<n>(h, xv));
                    }
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(&slot_empty[slot]);
                    if (++slot == kSlots) { slot = 0; slot_phase ^= 1; }
                }
            }
            if (!ok || !pipe::group_sync(p, pre_bar, pre_phase)) break;  // hp_buf is reused
            ++seg;
            if (pt == 0) *pre_done = seg;  // this segment's X has been re-read
        }
    } else if (warp == 14) {
        // ------------------------------------- coefficients (warp 14)
        // one lane per token (token_coeffs), 32 tokens per pass
        int seg = 0;
        ChunkIter it = segs;
        Segment sg;
        while (it.next(sg)) {
            const int t = sg.m;
            const int64_t row0 = static_cast<int64_t>(t) * kBM;
            const int valid = static_cast<int>(B - row0 < kBM ? B - row0 : kBM);
            const int nrows = clamp_rows(r0, r1, valid);
            const int rb = seg % kRowBufs;
            if (!pipe::wait(p, &rows_full[rb], (seg / kRowBufs) & 1)) break;
            for (int tk = lane; tk < nrows; tk += 32) {
                if (!in_range(508, row0 + r0 + tk, 1, B)) break;
                const float *yrow = rows_buf + (rb * kMaxRows + tk) * stride;
                float hp[n], hq[n], m[n][n];
                token_coeffs<n>(yrow, yrow[N], bias, a_pre, a_post, a_res, iters, hp, hq, m);
                store_token_coeffs<n>(row0 + r0 + tk, hp, hq, m, H_pre, H_post, H_res);
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&rows_empty[rb]);
            ++seg;
        }
    } else if (lane == 0) {
        // ------------------------------------------------ loader (warp 15)
        // X of a tile is in L2 once all its contributors have parked their
        // partials, which the tile's ticket counts.
        const uint64_t pol = ptx::policy_evict_first();  // the last read of this X
        int slot = 0;
        uint32_t slot_phase = 0;
        ChunkIter it = segs;
        Segment sg;
        bool ok = true;
        while (ok && it.next(sg)) {
            const int t = sg.m;
            const int64_t row0 = static_cast<int64_t>(t) * kBM;
            const int valid = static_cast<int>(B - row0 < kBM ? B - row0 : kBM);
            const int nrows = clamp_rows(r0, r1, valid);
            if (!wait_count(p, &tickets[t], fs.P)) {
                ok = false;
                break;
            }
            for (int tk = 0; tk < nrows && ok; ++tk) {
                const uint16_t *xrow = X + (row0 + r0 + tk) * K;
                const bool row_ok = in_range(509, row0 + r0 + tk, 1, B);
                for (int c0 = 0; c0 < C; c0 += W) {
                    const int wp = C - c0 < W ? C - c0 : W;
                    if (!pipe::wait(p, &slot_empty[slot], slot_phase ^ 1)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sl = slots + slot * kSlotBytes;
                    // a refused copy arrives without bytes: its reader skips it
                    const bool copy_ok = row_ok && in_range(510, c0, wp, C) &&
                                         in_range(511, 0, n * wp * 2, kSlotBytes);
                    ptx::mbar_arrive_expect_tx(&slot_full[slot],
                                               copy_ok ? static_cast<uint32_t>(n * wp * 2) : 0u);
                    if (copy_ok) {
#pragma unroll
                        for (int k = 0; k < n; ++k)
                            ptx::bulk_load(sl + k * wp * 2, xrow + static_cast<int64_t>(k) * C + c0,
                                           static_cast<uint32_t>(wp * 2), &slot_full[slot], pol);
                    }
                    if (++slot == kSlots) { slot = 0; slot_phase ^= 1; }
                }
            }
        }
        if (!ok) {
            // let the bulk copies in flight land before shared memory is released
            for (int s2 = 0; s2 < kSlots; ++s2) {
                volatile int never = 0;
                ptx::mbar_wait_bounded(&slot_full[s2], (s2 < slot ? slot_phase : slot_phase ^ 1),
                                       &never, p.limit_ns);
            }
        }
    }

    // lane 0 of the TMA, MMA and loader warps ran alone: reconverge every warp before
    // the CTA barrier, which needs whole warps
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::pdl_trigger();  // at the end, as in the standalone GEMM
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc<F::C::kTmemCols>(p.tmem_base);
    }
}

// Clears the tickets and reader counts of a call before its fused kernel runs.
__global__ void zero_counts_kernel(int *counts, int count)
{
    ptx::pdl_wait();
    ptx::pdl_trigger();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < count; i += gridDim.x * blockDim.x)
        counts[i] = 0;
}

// ------------------------------------------------------------------ host

struct Plan {
    bool ok = false;
    FSched fs{};
    int grid = 0;
    size_t ws_bytes = 0;
};

size_t counts_bytes(int m_tiles) { return (static_cast<size_t>(m_tiles) * 8 + 255) / 256 * 256; }

Plan make_plan(int64_t B, int n, int64_t C, int num_sms)
{
    Plan pl;
    const int64_t K = n * C;
    const int N = num_coeffs(n);
    const int64_t m_tiles = (B + kBM - 1) / kBM;
    const int kbt = static_cast<int>((K + kBK - 1) / kBK);
    const int64_t tile_bytes = static_cast<int64_t>(kBM) * K * 2;
    if (m_tiles < 2 || m_tiles > (int64_t{1} << 24)) return pl;
    // two or more partial buffers: a CTA parks tile t before it finishes the
    // tile before, so one buffer would have every CTA wait for the others
    const int nb = kLeadChunks + 1 < kMaxPartBufs ? kLeadChunks + 1 : kMaxPartBufs;
    if (kLeadChunks < 2 || nb < 2) return pl;
    for (int CH : {8, 4, 2, 1}) {
        const int P = num_sms / CH;
        if (CH > m_tiles || CH * tile_bytes > kChunkBytes || P < kBM / kMaxRows || kbt < P)
            continue;
        pl.fs = FSched{static_cast<int>(m_tiles), kbt, CH, P,
                       static_cast<int>((m_tiles + CH - 1) / CH), kLeadChunks, nb};
        pl.grid = CH * P;
        pl.ws_bytes = counts_bytes(static_cast<int>(m_tiles)) +
                      static_cast<size_t>(pl.fs.nb) * pl.grid * kBM * (N + 1) * sizeof(float);
        pl.ok = true;
        break;
    }
    return pl;
}

template <int n>
cudaError_t launch_n(const CUtensorMap &tx, const CUtensorMap &tw, const Plan &pl, int64_t B,
                     int64_t C, float a_pre, float a_post, float a_res, const float *bias,
                     int iters, const uint16_t *X, float *Y, float *r, float *H_pre,
                     float *H_post, float *H_res, uint16_t *F_pre, int *counts, float *partials,
                     cudaStream_t stream, int device)
{
    using F = FCfg<n>;
    static uint64_t configured = 0;
    static std::mutex mu;
    if (device < 64 && !((configured >> device) & 1)) {
        std::lock_guard<std::mutex> lock(mu);
        cudaError_t e = cudaFuncSetAttribute(fused_pre_kernel<n>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             F::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured |= 1ull << device;
    }
    const int m_tiles = pl.fs.m_tiles;
    // cooperative: the CTAs wait on one another, so all of them must be resident
    return launch_coop_pdl(fused_pre_kernel<n>, dim3(pl.grid), dim3(kThreads), F::kSmemBytes, stream,
                      tx, tw, B, static_cast<int>(n * C), static_cast<int>(C), pl.fs, a_pre,
                      a_post, a_res, bias, iters, X, Y, r, H_pre, H_post, H_res, F_pre, counts,
                      counts + m_tiles, partials, kWaitLimitNs);
}

}  // namespace

size_t fused_pre_workspace_bytes(int64_t B, int n, int64_t C, int num_sms)
{
    const Plan pl = make_plan(B, n, C, num_sms);
    return pl.ok ? pl.ws_bytes : 0;
}

bool fused_pre_eligible(int64_t B, int n, int64_t C, int num_sms)
{
    return make_plan(B, n, C, num_sms).ok;
}

cudaError_t launch_fused_pre(const uint16_t *X, const uint16_t *phi_t, float a_pre, float a_post,
                             float a_res, const float *bias, int iters, int64_t B, int n,
                             int64_t C, float *Y, float *r, float *H_pre, float *H_post,
                             float *H_res, uint16_t *F_pre, void *workspace, int num_sms,
                             cudaStream_t stream)
{
    const Plan pl = make_plan(B, n, C, num_sms);
    if (!pl.ok) return cudaErrorInvalidValue;
    const int N = num_coeffs(n);
    const int npad = (N + 15) / 16 * 16;
    CUtensorMap tx, tw;
    if (!make_tmap(&tx, X, static_cast<uint64_t>(n * C), static_cast<uint64_t>(B), kBM) ||
        !make_tmap(&tw, phi_t, static_cast<uint64_t>(n * C), static_cast<uint64_t>(N),
                   static_cast<uint32_t>(npad)))
        return cudaErrorInvalidValue;
    int *counts = static_cast<int *>(workspace);  // [m_tiles] tickets, then [m_tiles] readers
    float *partials = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                                counts_bytes(pl.fs.m_tiles));
    const int total = 2 * pl.fs.m_tiles;
    const int zb = total < 256 * 64 ? (total + 255) / 256 : 64;
    cudaError_t e = launch_pdl(zero_counts_kernel, dim3(zb), dim3(256), 0, stream, counts, total);
    if (e != cudaSuccess) return e;
    int device = 0;
    if ((e = cudaGetDevice(&device)) != cudaSuccess) return e;
    switch (n) {
#define MHC_CASE(k)                                                                             \
    case k:                                                                                     \
        return launch_n<k>(tx, tw, pl, B, C, a_pre, a_post, a_res, bias, iters, X, Y, r, H_pre, \
                           H_post, H_res, F_pre, counts, partials, stream, device);
        MHC_CASE(1) MHC_CASE(2) MHC_CASE(3) MHC_CASE(4) MHC_CASE(5) MHC_CASE(6) MHC_CASE(7)
        MHC_CASE(8)
#undef MHC_CASE
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t read_and_clear_fused_status(int *status)
{
    int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_fused_status, sizeof v);
    if (e != cudaSuccess) return e;
    if ((e = cudaMemcpyToSymbol(g_fused_status, &zero, sizeof zero)) != cudaSuccess) return e;
    *status = v;
    return cudaSuccess;
}

}  // namespace mhc
