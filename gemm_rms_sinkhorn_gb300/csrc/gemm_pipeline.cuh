// The X·φ + Σx² pipeline shared by the GEMM+RMS kernels (page "mHC 算法分析 &
// cutile 高效实现", §2.1, §2.2 and fusion §3.1):
//
//   TMA producer (1 thread)   128-token × 64-column boxes of X and NPAD × 64
//                             boxes of φᵀ, 128-byte swizzle, into a ring of
//                             shared-memory stages guarded by mbarriers;
//   MMA issuer (1 thread)     tcgen05.mma (M=128, N=NPAD, K=16; bf16 in, fp32
//                             accumulate) into a double-buffered TMEM accumulator;
//   square-sum (4 warps)      Σx² of each row from the same smem tiles (X leaves
//                             HBM once), handed over per segment through a
//                             double-buffered shared slot;
//   take_accumulator          the epilogue side: one segment's accumulator row
//                             (tcgen05.ld) and square sum into registers.
//
// A "segment" is one token tile (128 rows) and a contiguous range of 64-wide
// K blocks; every role walks the same sequence of segments, given by a
// segment iterator with `bool next(Segment &)`.  Every wait is bounded: on
// expiry the role raises the kernel's status word, sets the CTA's abort flag
// and returns, and the producer and the MMA issuer drain what they started.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "ptx.cuh"

namespace mhc {
namespace pipe {

constexpr int kBM = 128;            // tokens per tile (MMA M)
constexpr int kBK = 64;             // K elements per box: one 128-byte swizzle row
constexpr int kStatusTimeout = -5;  // MHC_ERR_TIMEOUT
constexpr int kBarrierBytes = 512;
constexpr int kSsBytes = 2 * kBM * 4;  // square-sum hand-over, double-buffered
constexpr int kBoxABytes = kBM * kBK * 2;  // one 128 × 64 bf16 box of X
// K elements per stage: a 128-byte swizzle row holds 64 bf16 or 128 e4m3
// values, so an 8-bit stage has the bf16 stage's bytes and layout.
template <bool kFp8>
constexpr int kKPerStage = kFp8 ? 2 * kBK : kBK;

// Stage geometry for MMA width NPAD (N padded to 16) and a shared-memory
// budget for the stage ring.
template <int NPAD, int BUDGET>
struct Cfg {
    static constexpr int kBoxA = kBoxABytes;
    static constexpr int kBoxB = NPAD * kBK * 2;  // one NPAD × 64 bf16 box of φᵀ
    static constexpr int kStageBytes = kBoxA + kBoxB;
    static constexpr int kStages = BUDGET / kStageBytes;
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kTmemCols =  // a power of two >= 32 holding both accumulators
        2 * NPAD <= 32 ? 32
                       : (2 * NPAD <= 64 ? 64 : (2 * NPAD <= 128 ? 128 : (2 * NPAD <= 256 ? 256 : 512)));
    static_assert(NPAD % 16 == 0 && NPAD >= 16 && NPAD <= 256, "MMA N for M=128");
    static_assert(kStageBytes % 1024 == 0, "stages keep 1024-byte alignment");
    static_assert(kStages >= 2 && kStages <= 32, "pipeline depth (one bit per stage)");
    static_assert((2 * kStages + 17) * 8 + 16 <= kBarrierBytes, "barrier area");
};

struct Segment {
    int m, k0, k1;  // token (row) tile, K-block range [k0, k1)
    int n = 0;      // column tile: rows [n·NPAD, (n+1)·NPAD) of the second operand
};

// Static stream-K schedule: the units (token tile, 64-wide K block), ordered
// tile-major, are split into `grid` equal contiguous ranges; CTA c owns units
// [lo(c), lo(c+1)).
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

// Pointers into one CTA's shared memory plus the per-kernel wait settings.
struct Pipe {
    uint8_t *stages;
    float *ss_buf;  // [2][kBM]
    uint64_t *full, *empty, *acc_full, *acc_empty, *ss_full, *ss_empty, *drain;
    uint64_t *extra;  // 8 more barriers for the kernel's own use
    uint32_t *tmem_holder;
    volatile int *abort;
    int *status;  // the kernel's device status word
    uint64_t limit_ns;
    int stages_n, stage_bytes, box_a;
    uint32_t tmem_base;
};

// Lays out [stage ring][square-sum slots][barriers + flags] from a
// 1024-aligned base.  Returns the first byte after the layout.
template <int NPAD, int BUDGET>
__device__ __forceinline__ uint8_t *carve(Pipe &p, uint8_t *base, int *status, uint64_t limit_ns)
{
    using C = Cfg<NPAD, BUDGET>;
    p.stages = base;
    p.ss_buf = reinterpret_cast<float *>(base + C::kRingBytes);
    uint64_t *b = reinterpret_cast<uint64_t *>(base + C::kRingBytes + kSsBytes);
    p.full = b;
    p.empty = b + C::kStages;
    p.acc_full = p.empty + C::kStages;  // [2] MMA -> epilogue
    p.acc_empty = p.acc_full + 2;       // [2] epilogue -> MMA
    p.ss_full = p.acc_empty + 2;        // [2] square-sum -> epilogue
    p.ss_empty = p.ss_full + 2;         // [2] epilogue -> square-sum
    p.drain = p.ss_empty + 2;           // MMA drain after an abort
    p.extra = p.drain + 1;              // [8]
    p.tmem_holder = reinterpret_cast<uint32_t *>(p.extra + 8);
    p.abort = reinterpret_cast<volatile int *>(p.tmem_holder + 1);
    p.status = status;
    p.limit_ns = limit_ns;
    p.stages_n = C::kStages;
    p.stage_bytes = C::kStageBytes;
    p.box_a = C::kBoxA;
    return base + C::kRingBytes + kSsBytes + kBarrierBytes;
}

// Thread 0 only, before the CTA-wide sync that precedes any use.
__device__ __forceinline__ void init_barriers(const Pipe &p)
{
    for (int s = 0; s < p.stages_n; ++s) {
        ptx::mbar_init(&p.full[s], 1);
        ptx::mbar_init(&p.empty[s], 1 + 4);  // MMA commit + one arrive per square-sum warp
    }
    for (int a = 0; a < 2; ++a) {
        ptx::mbar_init(&p.acc_full[a], 1);
        ptx::mbar_init(&p.acc_empty[a], 4);
        ptx::mbar_init(&p.ss_full[a], 4);
        ptx::mbar_init(&p.ss_empty[a], 4);
    }
    ptx::mbar_init(p.drain, 1);
    *p.abort = 0;
}

__device__ __forceinline__ void raise_timeout(const Pipe &p)
{
    *p.abort = 1;
    atomicExch(p.status, kStatusTimeout);
}

__device__ __forceinline__ bool wait(const Pipe &p, uint64_t *bar, uint32_t parity)
{
    if (ptx::mbar_wait_bounded(bar, parity, p.abort, p.limit_ns)) return true;
    raise_timeout(p);
    return false;
}

// ------------------------------------------------------------ producer
// One thread.  stall_stage >= 0 is a test hook: that stage (counted over the
// thread's whole run) is left unfilled so the consumers' waits run out.
template <int NPAD, typename It, bool kFp8 = false>
__device__ void producer(const Pipe &p, It it, const CUtensorMap *tm_x, const CUtensorMap *tm_w,
                         uint64_t pol_x, int64_t stall_stage)
{
    constexpr int kKS = kKPerStage<kFp8>;
    constexpr int kBoxA = kBoxABytes;
    const uint64_t pol_w = ptx::policy_evict_last();  // φ is re-read by every CTA
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0, issued_parity = 0;  // stages with a TMA issued, its phase
    int64_t count = 0;
    Segment sg;
    bool ok = true;
    while (ok && it.next(sg)) {
        for (int kb = sg.k0; kb < sg.k1; ++kb, ++count) {
            if (!wait(p, &p.empty[stage], phase ^ 1)) {
                ok = false;
                break;
            }
            if (count != stall_stage) {
                uint8_t *a = p.stages + stage * p.stage_bytes;
                ptx::mbar_arrive_expect_tx(&p.full[stage], p.stage_bytes);
                // boxes past K read as zeros
                ptx::tma_load_2d(a, tm_x, kb * kKS, sg.m * kBM, &p.full[stage], pol_x);
                ptx::tma_load_2d(a + kBoxA, tm_w, kb * kKS, sg.n * NPAD, &p.full[stage], pol_w);
                issued_mask |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            }
            if (++stage == p.stages_n) { stage = 0; phase ^= 1; }
        }
    }
    if (!ok) {
        // Let the copies already issued land before shared memory is released:
        // wait for the phase of each stage's last issue (already complete for
        // stages whose data was consumed).
        for (int s = 0; s < p.stages_n; ++s) {
            if (!((issued_mask >> s) & 1u)) continue;
            volatile int never = 0;
            ptx::mbar_wait_bounded(&p.full[s], (issued_parity >> s) & 1u, &never, p.limit_ns);
        }
    }
}

// ----------------------------------------------------------- MMA issuer
template <int NPAD, typename It, bool kFp8 = false>
__device__ void mma_issuer(const Pipe &p, It it)
{
    constexpr uint32_t idesc = kFp8 ? ptx::idesc_e4m3_f32(kBM, NPAD) : ptx::idesc_bf16_f32(kBM, NPAD);
    constexpr int kBoxA = kBoxABytes;
    int stage = 0;
    uint32_t phase = 0;
    int seg = 0;
    Segment sg;
    bool ok = true;
    while (ok && it.next(sg)) {
        const int acc = seg & 1;
        if (!wait(p, &p.acc_empty[acc], ((seg >> 1) & 1) ^ 1)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = p.tmem_base + static_cast<uint32_t>(acc * NPAD);
        for (int kb = sg.k0; kb < sg.k1; ++kb) {
            if (!wait(p, &p.full[stage], phase)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t a_addr = ptx::smem_u32(p.stages + stage * p.stage_bytes);
            const uint64_t a_desc = ptx::smem_desc_sw128(a_addr);
            const uint64_t b_desc = ptx::smem_desc_sw128(a_addr + kBoxA);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                // 32 bytes of K per instruction (16 bf16 or 32 e4m3): +2 in the
                // descriptor's address field
                const uint32_t accum = (kb > sg.k0 || kk > 0) ? 1u : 0u;
                if constexpr (kFp8)
                    ptx::mma_e4m3(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, idesc, accum);
                else
                    ptx::mma_bf16(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, idesc, accum);
            }
            ptx::mma_commit(&p.empty[stage]);  // frees the stage once these MMAs finish
            if (++stage == p.stages_n) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        ptx::mma_commit(&p.acc_full[acc]);
        ++seg;
    }
    // Before TMEM is released every MMA issued must have completed: a commit
    // arrives only after all prior tcgen05 ops of this thread.
    if (!ok || *p.abort) {
        ptx::mma_commit(p.drain);
        volatile int never = 0;
        ptx::mbar_wait_bounded(p.drain, 0, &never, p.limit_ns);
    }
}

// ----------------------------------------------------------- square-sum
// Warps w0..w0+3; thread `row` (0..127) sums row `row` of every stage.
template <int NPAD, typename It, bool kFp8 = false>
__device__ void square_sum(const Pipe &p, It it, int row, int lane)
{
    int stage = 0;
    uint32_t phase = 0;
    int seg = 0;
    Segment sg;
    bool ok = true;
    while (ok && it.next(sg)) {
        float ss0 = 0.f, ss1 = 0.f, ss2 = 0.f, ss3 = 0.f;
        for (int kb = sg.k0; kb < sg.k1; ++kb) {
            if (!wait(p, &p.full[stage], phase)) {
                ok = false;
                break;
            }
            const uint8_t *arow = p.stages + stage * p.stage_bytes + row * 128;
            // 16-byte chunk j of the row lives at chunk (j ^ row%8) (128-byte
            // swizzle); a row sum needs every chunk once, in any order.
            uint4 row_v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                row_v[j] = *reinterpret_cast<const uint4 *>(arow + ((j ^ (row & 7)) << 4));
            const auto release = [&] {
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&p.empty[stage]);  // release: orders the loads
                if (++stage == p.stages_n) { stage = 0; phase ^= 1; }
            };
            // e4m3 rows cost about three times the arithmetic of bf16 rows: their
            // stage goes back before it, so the ring refills meanwhile (measured
            // at B=16384, n=4, C=7168: 86.8 -> 85.6 us; the same order made the
            // bf16 GEMM 1 us slower, so bf16 keeps arithmetic-then-release).
            if constexpr (kFp8) release();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint4 v = row_v[j];
                if constexpr (kFp8) {
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        e4m3x2_square_add(w[h], ss0, ss1);
                        e4m3x2_square_add(w[h] >> 16, ss2, ss3);
                    }
                } else {
                    const float a0 = bf16_lo(v.x), a1 = bf16_hi(v.x), a2 = bf16_lo(v.y);
                    const float a3 = bf16_hi(v.y), a4 = bf16_lo(v.z), a5 = bf16_hi(v.z);
                    const float a6 = bf16_lo(v.w), a7 = bf16_hi(v.w);
                    ss0 = fmaf(a0, a0, ss0); ss1 = fmaf(a1, a1, ss1);
                    ss2 = fmaf(a2, a2, ss2); ss3 = fmaf(a3, a3, ss3);
                    ss0 = fmaf(a4, a4, ss0); ss1 = fmaf(a5, a5, ss1);
                    ss2 = fmaf(a6, a6, ss2); ss3 = fmaf(a7, a7, ss3);
                }
            }
            if constexpr (!kFp8) release();
        }
        if (!ok) break;
        // hand the segment's row sums to the epilogue
        const int buf = seg & 1;
        if (!wait(p, &p.ss_empty[buf], ((seg >> 1) & 1) ^ 1)) break;
        p.ss_buf[buf * kBM + row] = (ss0 + ss1) + (ss2 + ss3);
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&p.ss_full[buf]);
        ++seg;
    }
}

// ------------------------------------------------------- epilogue side
// Called by the 4 epilogue warps for their `seg`-th segment: thread `lane` of
// the warp with TMEM lane quarter q receives row q*32+lane of the
// accumulator and its square sum, and both buffers are handed back.
// Returns false when a wait ran out.
template <int NPAD>
__device__ bool take_accumulator(const Pipe &p, int seg, int q, int lane, float (&v)[NPAD],
                                 float &ss)
{
    const int acc = seg & 1;
    const uint32_t par = (seg >> 1) & 1;
    if (!wait(p, &p.acc_full[acc], par)) return false;
    ptx::tc_fence_after();
    const uint32_t taddr = p.tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
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
    if (lane == 0) ptx::mbar_arrive(&p.acc_empty[acc]);
    if (!wait(p, &p.ss_full[acc], par)) return false;
    ss = p.ss_buf[acc * kBM + q * 32 + lane];
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&p.ss_empty[acc]);
    return true;
}

// As take_accumulator, for wide accumulators: the row leaves TMEM 32 columns at
// a time and fn(chunk, v) consumes each chunk (columns chunk·32 .. +31; past
// NPAD the values are zero) before the next is loaded.
template <int NPAD, typename F>
__device__ bool take_accumulator_chunked(const Pipe &p, int seg, int q, int lane, float &ss,
                                         F &&fn)
{
    const int acc = seg & 1;
    const uint32_t par = (seg >> 1) & 1;
    if (!wait(p, &p.acc_full[acc], par)) return false;
    ptx::tc_fence_after();
    const uint32_t taddr = p.tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                           static_cast<uint32_t>(acc * NPAD);
#pragma unroll 1
    for (int c = 0; c < (NPAD + 31) / 32; ++c) {
        float v[32], t[16];
        ptx::tmem_ld_16(taddr + c * 32, t);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = t[e];
        if (c * 32 + 16 < NPAD) {
            ptx::tmem_ld_16(taddr + c * 32 + 16, t);
#pragma unroll
            for (int e = 0; e < 16; ++e) v[16 + e] = t[e];
        } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) v[16 + e] = 0.f;
        }
        ptx::tmem_ld_wait();
        fn(c, v);
        __syncwarp();  // the next tcgen05.ld is warp-collective
    }
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&p.acc_empty[acc]);
    if (!wait(p, &p.ss_full[acc], par)) return false;
    ss = p.ss_buf[acc * kBM + q * 32 + lane];
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&p.ss_empty[acc]);
    return true;
}

// Group barrier of `count` threads on an mbarrier (bounded like every wait).
__device__ __forceinline__ bool group_sync(const Pipe &p, uint64_t *bar, uint32_t &phase)
{
    ptx::mbar_arrive(bar);
    const bool ok = wait(p, bar, phase);
    phase ^= 1;
    return ok;
}

}  // namespace pipe
}  // namespace mhc
