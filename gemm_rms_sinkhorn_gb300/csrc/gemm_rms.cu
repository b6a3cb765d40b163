// Step 1 of the mHC forward: the skinny projection GEMM fused with the RMS
// reduction (page "mHC 算法分析 & cutile 高效实现", §2.1, §2.2, fusion §3.1;
// split-K motivation §5.1).
//
//   Y[b][k] = Σ_q X[b][q]·φ[q][k]    r[b] = sqrt(Σ_q X[b][q]² / K)
//
// Design (sm_103a):
//   * Work unit = one 128-token × (64·KB)-K block, one pipeline stage of KB
//     consecutive 64-column boxes (KB = kKB).  Units are ordered tile-major
//     (all K blocks of token tile 0, then tile 1, ...) and split into equal
//     contiguous ranges, one per persistent CTA (stream-K), so every SM gets
//     the same number of units whatever B and K are.  N is tiny (24 or 80),
//     so output tiling alone would leave most SMs idle (§5.1).
//   * Warp 0 streams X and φᵀ tiles with TMA (128-byte swizzle) through a
//     multi-stage mbarrier ring.  Warp 1 issues tcgen05.mma (M=128,
//     N=NPAD, K=16, bf16 in, fp32 accumulate) into a double-buffered TMEM
//     accumulator.  Warps 2-5 sum x² for their 32 rows straight from the same
//     shared-memory tiles (X is read from HBM once) and hand each segment's
//     sums over through a double-buffered shared slot.  Warps 6-9 run the
//     epilogue (tcgen05.ld of the accumulator, partial sums, the fixed-order
//     reduction), so the stage consumers never wait on epilogue work.
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

#include "mhc_internal.h"
#include "ptx.cuh"

namespace mhc {
namespace {

constexpr int kBM = 128;       // tokens per tile (MMA M)
constexpr int kBK = 64;        // K elements per box: one 128-byte swizzle row
constexpr int kKB = 1;         // boxes per stage (2 and 4 measured no faster on GB300)
constexpr int kThreads = 320;  // 10 warps: TMA, MMA, 4 × square-sum, 4 × epilogue
constexpr int kEpiThreads = 128;
constexpr int kReduceItems = 4;   // outputs per thread per round of the fixed-order sum
constexpr int kReduceBatch = 8;   // contributors loaded per batch: 32 loads in flight
constexpr int kStatusTimeout = -5;                // MHC_ERR_TIMEOUT

__device__ int g_device_status;

// NPAD: MMA N (N padded to 16); KB: 64-column boxes per stage; CPS: CTAs
// meant to share one SM (shared memory split between them; 1 is used, 2
// measured slower).
template <int NPAD, int KB, int CPS>
struct Cfg {
    static constexpr int kBoxA = kBM * kBK * 2;    // one 128 × 64 bf16 box of X
    static constexpr int kBoxB = NPAD * kBK * 2;   // one NPAD × 64 bf16 box of φᵀ
    static constexpr int kABytes = KB * kBoxA;     // A boxes of a stage, then its B boxes
    static constexpr int kStageBytes = KB * (kBoxA + kBoxB);
    static constexpr int kStages = (CPS == 1 ? 200 * 1024 : 100 * 1024) / kStageBytes;
    static constexpr int kTmemCols =
        2 * NPAD <= 32 ? 32 : (2 * NPAD <= 64 ? 64 : (2 * NPAD <= 128 ? 128 : 256));
    static constexpr int kBarrierBytes = 512;
    static constexpr int kSsBytes = 2 * kBM * 4;  // square-sum hand-over, double-buffered
    static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kSsBytes + kBarrierBytes;
    static_assert(NPAD % 16 == 0 && NPAD >= 16 && NPAD <= 256, "MMA N for M=128");
    static_assert(kStageBytes % 1024 == 0, "stages keep 1024-byte alignment");
    static_assert(kStages >= 2 && kStages <= 32, "pipeline depth (one bit per stage)");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
    static_assert((2 * kStages + 10) * 8 + 16 <= kBarrierBytes, "barrier area");
};

// Static stream-K schedule: CTA c owns units [lo(c), lo(c+1)).
struct Sched {
    int64_t total;  // m_tiles * kbt
    int kbt;        // K blocks per token tile
    int m_tiles;
    int grid;
    __host__ __device__ int64_t lo(int c) const { return total * c / grid; }
    // The CTA whose range holds unit u.
    __host__ __device__ int owner(int64_t u) const {
        return static_cast<int>(((u + 1) * grid - 1) / total);
    }
};

struct Segment {
    int m, k0, k1;
};

// Walks the segments (one token tile, a contiguous K-block range) of a CTA.
struct SegIter {
    int64_t u, end;
    int kbt;
    __device__ bool next(Segment &s) {
        if (u >= end) return false;
        s.m = static_cast<int>(u / kbt);
        s.k0 = static_cast<int>(u - static_cast<int64_t>(s.m) * kbt);
        int64_t left = end - u;
        s.k1 = left < kbt - s.k0 ? s.k0 + static_cast<int>(left) : kbt;
        u += s.k1 - s.k0;
        return true;
    }
};

// Group barrier of the 128 epilogue threads on an mbarrier, so that the wait
// is bounded like every other wait in the kernel.
__device__ __forceinline__ bool epi_sync(uint64_t *bar, uint32_t &phase, volatile int *abort_flag,
                                         uint64_t limit_ns) {
    ptx::mbar_arrive(bar);
    const bool ok = ptx::mbar_wait_bounded(bar, phase, abort_flag, limit_ns);
    phase ^= 1;
    return ok;
}

__device__ __forceinline__ void raise_timeout(volatile int *abort_flag) {
    *abort_flag = 1;
    atomicExch(&g_device_status, kStatusTimeout);
}

template <int NPAD, int KB, int CPS>
__global__ void __launch_bounds__(kThreads, 1)
gemm_rms_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                int64_t B, int N, int K, Sched sch, float *__restrict__ Y, float *__restrict__ r,
                int *__restrict__ tile_tickets, float *__restrict__ partials,
                uint64_t wait_limit_ns, int64_t stall_stage)
{
    using C = Cfg<NPAD, KB, CPS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float *ss_buf = reinterpret_cast<float *>(smem + C::kStages * C::kStageBytes);  // [2][128]
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kStages * C::kStageBytes + C::kSsBytes);
    uint64_t *empty = full + C::kStages;
    uint64_t *acc_full = empty + C::kStages;  // [2] MMA -> epilogue
    uint64_t *acc_empty = acc_full + 2;       // [2] epilogue -> MMA
    uint64_t *ss_full = acc_empty + 2;        // [2] square-sum -> epilogue
    uint64_t *ss_empty = ss_full + 2;         // [2] epilogue -> square-sum
    uint64_t *epi_bar = ss_empty + 2;         // epilogue group barrier
    uint64_t *drain_bar = epi_bar + 1;        // MMA drain after an abort
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain_bar + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    volatile int *is_last = reinterpret_cast<volatile int *>(tmem_holder + 2);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1 + 4);  // MMA commit + one arrive per square-sum warp
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&acc_full[a], 1);
            ptx::mbar_init(&acc_empty[a], 4);
            ptx::mbar_init(&ss_full[a], 4);
            ptx::mbar_init(&ss_empty[a], 4);
        }
        ptx::mbar_init(epi_bar, kEpiThreads);
        ptx::mbar_init(drain_bar, 1);
        *abort_flag = 0;
        *is_last = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tm_x);
        ptx::prefetch_tensormap(&tm_w);
    }
    if (warp == 1) ptx::tmem_alloc<C::kTmemCols>(tmem_holder);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // everything above is on-chip set-up; global memory is touched only after
    // the previous kernel in the stream has completed
    ptx::pdl_wait();

    const int64_t u_begin = sch.lo(cta), u_end = sch.lo(cta + 1);

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_x = ptx::policy_evict_first();  // X streams through once
            const uint64_t pol_w = ptx::policy_evict_last();   // φ is re-read by every CTA
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, issued_parity = 0;  // stages with a TMA issued, its phase
            int64_t count = 0;
            SegIter it{u_begin, u_end, sch.kbt};
            Segment sg;
            bool ok = true;
            while (ok && it.next(sg)) {
                for (int kb = sg.k0; kb < sg.k1; ++kb, ++count) {
                    if (!ptx::mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag,
                                                wait_limit_ns)) {
                        raise_timeout(abort_flag);
                        ok = false;
                        break;
                    }
                    // test hook: CTA 0 leaves one stage unfilled, so its consumers'
                    // bounded waits run out (stall_stage < 0 in normal calls)
                    if (!(cta == 0 && count == stall_stage)) {
                        uint8_t *a = smem + stage * C::kStageBytes;
                        ptx::mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
#pragma unroll
                        for (int b = 0; b < KB; ++b)  // boxes past K read as zeros
                            ptx::tma_load_2d(a + b * C::kBoxA, &tm_x, (kb * KB + b) * kBK,
                                             sg.m * kBM, &full[stage], pol_x);
#pragma unroll
                        for (int b = 0; b < KB; ++b)
                            ptx::tma_load_2d(a + C::kABytes + b * C::kBoxB, &tm_w,
                                             (kb * KB + b) * kBK, 0, &full[stage], pol_w);
                        issued_mask |= 1u << stage;
                        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == C::kStages) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) {
                // Let the copies already issued land before shared memory is released:
                // wait for the phase of each stage's last issue (already complete for
                // stages whose data was consumed).
                for (int s2 = 0; s2 < C::kStages; ++s2) {
                    if (!((issued_mask >> s2) & 1u)) continue;
                    volatile int never = 0;
                    ptx::mbar_wait_bounded(&full[s2], (issued_parity >> s2) & 1u, &never,
                                           wait_limit_ns);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_bf16_f32(kBM, NPAD);
            int stage = 0;
            uint32_t phase = 0;
            int seg = 0;
            SegIter it{u_begin, u_end, sch.kbt};
            Segment sg;
            bool ok = true;
            while (ok && it.next(sg)) {
                const int acc = seg & 1;
                if (!ptx::mbar_wait_bounded(&acc_empty[acc], ((seg >> 1) & 1) ^ 1, abort_flag,
                                            wait_limit_ns)) {
                    raise_timeout(abort_flag);
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * NPAD);
                for (int kb = sg.k0; kb < sg.k1; ++kb) {
                    if (!ptx::mbar_wait_bounded(&full[stage], phase, abort_flag, wait_limit_ns)) {
                        raise_timeout(abort_flag);
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a_addr = ptx::smem_u32(smem + stage * C::kStageBytes);
#pragma unroll
                    for (int b = 0; b < KB; ++b) {
                        const uint64_t a_desc = ptx::smem_desc_sw128(a_addr + b * C::kBoxA);
                        const uint64_t b_desc =
                            ptx::smem_desc_sw128(a_addr + C::kABytes + b * C::kBoxB);
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk) {
                            // advancing K by 16 bf16 = 32 bytes inside the swizzle row
                            ptx::mma_bf16(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, idesc,
                                          (kb > sg.k0 || b > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    ptx::mma_commit(&empty[stage]);  // frees the stage once these MMAs finish
                    if (++stage == C::kStages) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                ptx::mma_commit(&acc_full[acc]);
                ++seg;
            }
            // Before TMEM is released every MMA issued must have completed: a
            // commit arrives only after all prior tcgen05 ops of this thread.
            if (!ok || *abort_flag) {
                ptx::mma_commit(drain_bar);
                volatile int never = 0;
                ptx::mbar_wait_bounded(drain_bar, 0, &never, wait_limit_ns);
            }
        }
    } else if (warp < 6) {
        // ---------------------------------------- square-sum (warps 2..5)
        const int row = (warp - 2) * 32 + lane;
        int stage = 0;
        uint32_t phase = 0;
        int seg = 0;
        SegIter it{u_begin, u_end, sch.kbt};
        Segment sg;
        bool ok = true;
        while (ok && it.next(sg)) {
            float ss0 = 0.f, ss1 = 0.f, ss2 = 0.f, ss3 = 0.f;
            for (int kb = sg.k0; kb < sg.k1; ++kb) {
                if (!ptx::mbar_wait_bounded(&full[stage], phase, abort_flag, wait_limit_ns)) {
                    raise_timeout(abort_flag);
                    ok = false;
                    break;
                }
                const uint8_t *arow = smem + stage * C::kStageBytes + row * 128;
#pragma unroll
                for (int j = 0; j < 8 * KB; ++j) {
                    // 16-byte chunk j%8 of the row in box j/8 lives at chunk (j ^ row%8)
                    // (128-byte swizzle); a row sum needs every chunk once, in any order.
                    const uint4 v = *reinterpret_cast<const uint4 *>(
                        arow + (j >> 3) * C::kBoxA + (((j & 7) ^ (row & 7)) << 4));
                    float a0 = bf16_lo(v.x), a1 = bf16_hi(v.x), a2 = bf16_lo(v.y), a3 = bf16_hi(v.y);
                    float a4 = bf16_lo(v.z), a5 = bf16_hi(v.z), a6 = bf16_lo(v.w), a7 = bf16_hi(v.w);
                    ss0 = fmaf(a0, a0, ss0); ss1 = fmaf(a1, a1, ss1);
                    ss2 = fmaf(a2, a2, ss2); ss3 = fmaf(a3, a3, ss3);
                    ss0 = fmaf(a4, a4, ss0); ss1 = fmaf(a5, a5, ss1);
                    ss2 = fmaf(a6, a6, ss2); ss3 = fmaf(a7, a7, ss3);
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&empty[stage]);
                if (++stage == C::kStages) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
            // hand the segment's row sums to the epilogue warps
            const int buf = seg & 1;
            if (!ptx::mbar_wait_bounded(&ss_empty[buf], ((seg >> 1) & 1) ^ 1, abort_flag,
                                        wait_limit_ns)) {
                raise_timeout(abort_flag);
                break;
            }
            ss_buf[buf * kBM + row] = (ss0 + ss1) + (ss2 + ss3);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&ss_full[buf]);
            ++seg;
        }
    } else {
        // ----------------------------------------------- epilogue (warps 6..9)
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        const int et = threadIdx.x - 192;  // 0..127 within the epilogue group
        uint32_t epi_phase = 0;
        int seg = 0;
        SegIter it{u_begin, u_end, sch.kbt};
        Segment sg;
        while (it.next(sg)) {
            // accumulator and square-sum of this segment -> registers
            const int acc = seg & 1;
            const uint32_t par = (seg >> 1) & 1;
            if (!ptx::mbar_wait_bounded(&acc_full[acc], par, abort_flag, wait_limit_ns)) {
                raise_timeout(abort_flag);
                break;
            }
            ptx::tc_fence_after();
            float v[NPAD];
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * NPAD);
#pragma unroll
            for (int j = 0; j < NPAD / 16; ++j) {
                float t[16];
                ptx::tmem_ld_16(taddr + j * 16, t);
#pragma unroll
                for (int e = 0; e < 16; ++e) v[j * 16 + e] = t[e];
            }
            ptx::tmem_ld_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&acc_empty[acc]);
            if (!ptx::mbar_wait_bounded(&ss_full[acc], par, abort_flag, wait_limit_ns)) {
                raise_timeout(abort_flag);
                break;
            }
            const float ss = ss_buf[acc * kBM + row];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&ss_empty[acc]);
            ++seg;

            const int64_t row0 = static_cast<int64_t>(sg.m) * kBM;
            const int64_t grow = row0 + row;
            if (sg.k0 == 0 && sg.k1 == sch.kbt) {
                // the whole K range of this tile is ours: write the result
                if (grow < B) {
                    float *y = Y + grow * N;
#pragma unroll
                    for (int j = 0; j < NPAD; ++j)
                        if (j < N) y[j] = v[j];
                    r[grow] = sqrtf(ss / static_cast<float>(K));
                }
                continue;
            }
            // partial: park [row][N+1] in this (cta, tile) slot, then take a ticket
            const int stride = N + 1;
            float *mine = partials + static_cast<int64_t>(cta + sg.m) * kBM * stride;
            if (grow < B) {
#pragma unroll
                for (int j = 0; j < NPAD; ++j)
                    if (j < N) mine[row * stride + j] = v[j];
                mine[row * stride + N] = ss;
            }
            __threadfence();
            if (!epi_sync(epi_bar, epi_phase, abort_flag, wait_limit_ns)) { raise_timeout(abort_flag); break; }
            const int first = sch.owner(static_cast<int64_t>(sg.m) * sch.kbt);
            const int last = sch.owner(static_cast<int64_t>(sg.m + 1) * sch.kbt - 1);
            if (et == 0) {
                const int prev = atomicAdd(&tile_tickets[sg.m], 1);
                *is_last = (prev == last - first);
            }
            if (!epi_sync(epi_bar, epi_phase, abort_flag, wait_limit_ns)) { raise_timeout(abort_flag); break; }
            if (*is_last) {
                __threadfence();
                // fixed-order sum over the contributors first..last: a batch of
                // contributors x items is loaded before it is added, in order
                const int64_t rows = (B - row0) < kBM ? (B - row0) : kBM;
                const int items = static_cast<int>(rows) * stride;
                const float *p0 = partials + static_cast<int64_t>(first + sg.m) * kBM * stride;
                const int64_t slot_stride = static_cast<int64_t>(kBM) * stride;
                const int nc = last - first + 1;
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
                                vb[c][u] = (c0 + c < nc && i < items)
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
                        const int rr = i / stride, cc = i - rr * stride;
                        if (cc < N)
                            Y[(row0 + rr) * N + cc] = acc_s[u];
                        else
                            r[row0 + rr] = sqrtf(acc_s[u] / static_cast<float>(K));
                    }
                }
                if (et == 0) tile_tickets[sg.m] = 0;
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    // Let the next kernel launch only now: CTAs of a dependent kernel that sit
    // resident in pdl_wait next to this one for its whole run slow it down
    // (measured: +13% at B=16384), while a trigger at the end still hides
    // the launch latency.
    ptx::pdl_trigger();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc<C::kTmemCols>(tmem_base);
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

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
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

// 2-D bf16 tensor [rows][cols] (cols contiguous), box [box_rows][64], 128-byte swizzle.
bool make_tmap(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_rows)
{
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
    cuuint32_t estr[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int npad_of(int n)
{
    const int N = num_coeffs(n);
    return (N + 15) / 16 * 16;
}

// Grid: one CTA per SM, but no more than 32 contributors per token tile (the
// last arriver's fixed-order sum grows with the fan-in) and at least one
// stage of K per CTA.
Sched make_sched(int64_t B, int n, int64_t C, int num_sms)
{
    Sched s;
    s.m_tiles = static_cast<int>((B + kBM - 1) / kBM);
    s.kbt = static_cast<int>((n * C + kBK * kKB - 1) / (kBK * kKB));
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
};

template <int NPAD, int KB, int CPS>
cudaError_t launch_cfg(const LaunchArgs &a)
{
    using Cf = Cfg<NPAD, KB, CPS>;
    static uint64_t configured = 0;  // one bit per device
    static std::mutex mu;
    if (a.device < 64 && !((configured >> a.device) & 1)) {
        std::lock_guard<std::mutex> lock(mu);
        cudaError_t e = cudaFuncSetAttribute(gemm_rms_kernel<NPAD, KB, CPS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Cf::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured |= 1ull << a.device;
    }
    return launch_pdl(gemm_rms_kernel<NPAD, KB, CPS>, dim3(a.s.grid), dim3(kThreads),
                      Cf::kSmemBytes, a.stream, *a.tx, *a.tw, a.B, a.N, a.K, a.s, a.Y, a.r,
                      a.tickets, a.partials, a.wait_limit_ns, a.stall_stage);
}

cudaError_t dispatch(int npad, const LaunchArgs &a)
{
    switch (npad) {
    case 16: return launch_cfg<16, kKB, 1>(a);
    case 32: return launch_cfg<32, kKB, 1>(a);
    case 48: return launch_cfg<48, kKB, 1>(a);
    case 64: return launch_cfg<64, kKB, 1>(a);
    case 80: return launch_cfg<80, kKB, 1>(a);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t gemm_rms_workspace_bytes(int64_t B, int n, int64_t C, int num_sms)
{
    if (B <= 0) return 0;
    const Sched s = make_sched(B, n, C, num_sms);
    const int N = num_coeffs(n);
    const size_t slots = static_cast<size_t>(s.grid) + s.m_tiles;
    return tickets_bytes(s.m_tiles) + slots * kBM * (N + 1) * sizeof(float);
}

cudaError_t launch_gemm_rms(const uint16_t *X, const uint16_t *phi_t, int64_t B, int n,
                            int64_t C, float *Y, float *r, void *workspace, int num_sms,
                            cudaStream_t stream, uint64_t wait_limit_ns, int64_t stall_stage)
{
    const int N = num_coeffs(n);
    const int64_t K = n * C;
    const Sched s = make_sched(B, n, C, num_sms);
    CUtensorMap tx, tw;
    const int npad = npad_of(n);
    if (!make_tmap(&tx, X, static_cast<uint64_t>(K), static_cast<uint64_t>(B), kBM) ||
        !make_tmap(&tw, phi_t, static_cast<uint64_t>(K), static_cast<uint64_t>(N),
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
                       device, wait_limit_ns, stall_stage};
    return dispatch(npad, a);
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
