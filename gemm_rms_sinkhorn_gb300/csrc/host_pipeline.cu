// The forward over host-resident activations (mhc_forward_host): the batch
// goes through the device in chunks of tokens (ramped at both ends, see
// chunk_sizes), and the copy of chunk k+1 to
// the device, the forward of chunk k and the copy of chunk k-1's outputs back
// overlap on three streams, so a step costs about the slower copy direction
// rather than the sum of both copies and the compute.  Tokens are independent
// in every step of the forward (page "mHC 算法分析 & cutile 高效实现", §2.3), so
// chunking changes no result beyond the split-K order inside each chunk.
//
// Each chunk's bf16 buffers (X, which X_next overwrites in place, F_out and
// F_pre) rotate over kHostSlots = 3 slots of the caller's device scratch; the
// small fp32 outputs (Y, r, H) of the whole batch stay on the device until
// the end and go back in one copy each; events order the reuse of a slot after its outputs have left the
// device.  With three slots the loop copy-in -> forward -> copy-out -> next
// copy-in into the same slot spans three chunks, so neither copy direction
// waits on the other in the steady state.
// The copy streams and events are created once per device and kept.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <vector>

#include "mhc.h"
#include "mhc_internal.h"
#include "mhc_testing.h"

namespace mhc {
namespace {

constexpr int kSlots = kHostSlots;

struct HostRuntime {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr;
    cudaEvent_t loaded[kSlots] = {}, computed[kSlots] = {}, drained[kSlots] = {};
};

constexpr int kMaxDevices = 64;
HostRuntime g_rt[kMaxDevices];
std::mutex g_rt_mu[kMaxDevices];

cudaError_t init_runtime(HostRuntime &rt)
{
    if (rt.ready) return cudaSuccess;
    cudaError_t e;
    if ((e = cudaStreamCreateWithFlags(&rt.h2d, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&rt.d2h, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&rt.start, cudaEventDisableTiming)) != cudaSuccess) return e;
    for (int s = 0; s < kSlots; ++s) {
        if ((e = cudaEventCreateWithFlags(&rt.loaded[s], cudaEventDisableTiming)) != cudaSuccess)
            return e;
        if ((e = cudaEventCreateWithFlags(&rt.computed[s], cudaEventDisableTiming)) != cudaSuccess)
            return e;
        if ((e = cudaEventCreateWithFlags(&rt.drained[s], cudaEventDisableTiming)) != cudaSuccess)
            return e;
    }
    rt.ready = true;
    return cudaSuccess;
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

// Token count of each chunk, in order, for chunks of at most `full` tokens.
// The first copy in and the last copy out overlap nothing, so the schedule
// ramps up (full/4, full/2, then full chunks) and back down (full/2, full/4)
// at the end; a batch too small for the ramp goes in equal chunks of full/4
// tokens (at least 1), the last possibly shorter.
std::vector<int64_t> chunk_sizes(int64_t B, int64_t full)
{
    const int64_t ramp[2] = {full / 4, full / 2};
    std::vector<int64_t> out;
    auto push = [&](int64_t v) {
        if (v > 0) out.push_back(v);
    };
    if (B < 2 * (ramp[0] + ramp[1]) + full) {
        const int64_t step = ramp[0] > 0 ? ramp[0] : 1;
        for (int64_t t = 0; t < B; t += step) push(B - t < step ? B - t : step);
        return out;
    }
    push(ramp[0]);
    push(ramp[1]);
    int64_t mid = B - 2 * (ramp[0] + ramp[1]);
    for (; mid > 0; mid -= full) push(mid < full ? mid : full);
    push(ramp[1]);
    push(ramp[0]);
    return out;
}

}  // namespace

HostChunkLayout host_chunk_layout(int64_t B, int n, int64_t C, int num_sms)
{
    HostChunkLayout L{};
    const int64_t Bc = B < kHostChunkTokens ? B : kHostChunkTokens;
    const int N = num_coeffs(n);
    L.chunk_tokens = Bc;
    // per slot: the chunk's bf16 activations
    L.x = align256(static_cast<size_t>(Bc) * n * C * 2);
    L.f_out = align256(static_cast<size_t>(Bc) * C * 2);
    L.f_pre = L.f_out;
    L.slot = L.x + L.f_out + L.f_pre;
    // for the whole batch: the small fp32 outputs, copied back once at the end
    // (a few bytes a token; a copy costs microseconds however small it is)
    L.y = align256(static_cast<size_t>(B) * N * 4);
    L.r = align256(static_cast<size_t>(B) * 4);
    L.h_pre = align256(static_cast<size_t>(B) * n * 4);
    L.h_post = L.h_pre;
    L.h_res = align256(static_cast<size_t>(B) * n * n * 4);
    L.workspace = align256(forward_workspace_bytes(Bc, n, C, num_sms));
    L.total = kHostSlots * L.slot + L.y + L.r + L.h_pre + L.h_post + L.h_res + L.workspace;
    return L;
}

cudaError_t run_forward_host(const uint16_t *X, const uint16_t *phi_t, const uint16_t *F_out,
                             float a_pre, float a_post, float a_res, const float *bias, int iters,
                             int64_t B, int n, int64_t C, float *Y, float *r, float *H_pre,
                             float *H_post, float *H_res, uint16_t *F_pre, uint16_t *X_next,
                             void *scratch, int num_sms, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_rt_mu[dev]);  // one enqueue at a time per device
    HostRuntime &rt = g_rt[dev];
    if ((e = init_runtime(rt)) != cudaSuccess) return e;

    const HostChunkLayout L = host_chunk_layout(B, n, C, num_sms);
    const int N = num_coeffs(n);
    const int64_t K = n * C;
    uint8_t *base = static_cast<uint8_t *>(scratch);
    float *gy = reinterpret_cast<float *>(base + kSlots * L.slot);
    float *gr = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(gy) + L.y);
    float *ghp = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(gr) + L.r);
    float *ghq = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(ghp) + L.h_pre);
    float *ghr = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(ghq) + L.h_post);
    void *ws = reinterpret_cast<uint8_t *>(ghr) + L.h_res;

    // everything below is ordered after the caller's earlier work on `stream`
    if ((e = cudaEventRecord(rt.start, stream)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(rt.h2d, rt.start, 0)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(rt.d2h, rt.start, 0)) != cudaSuccess) return e;

    const std::vector<int64_t> sizes = chunk_sizes(B, L.chunk_tokens);
    const int64_t chunks = static_cast<int64_t>(sizes.size());
    int64_t t0 = 0;
    for (int64_t k = 0; k < chunks; t0 += sizes[k], ++k) {
        const int s = static_cast<int>(k % kSlots);
        const int64_t bc = sizes[k];
        uint8_t *p = base + s * L.slot;
        uint16_t *dx = reinterpret_cast<uint16_t *>(p);
        uint16_t *df = reinterpret_cast<uint16_t *>(p + L.x);
        uint16_t *dfp = reinterpret_cast<uint16_t *>(p + L.x + L.f_out);

        // inputs of chunk k, once the outputs of chunk k - kSlots have left the slot
        if (k >= kSlots && (e = cudaStreamWaitEvent(rt.h2d, rt.drained[s], 0)) != cudaSuccess)
            return e;
        if ((e = cudaMemcpyAsync(dx, X + t0 * K, bc * K * 2, cudaMemcpyHostToDevice, rt.h2d)) !=
            cudaSuccess)
            return e;
        if ((e = cudaMemcpyAsync(df, F_out + t0 * C, bc * C * 2, cudaMemcpyHostToDevice,
                                 rt.h2d)) != cudaSuccess)
            return e;
        if ((e = cudaEventRecord(rt.loaded[s], rt.h2d)) != cudaSuccess) return e;

        // the forward of chunk k on the caller's stream, X_next in place over X
        if ((e = cudaStreamWaitEvent(stream, rt.loaded[s], 0)) != cudaSuccess) return e;
        if ((e = run_forward_device(dx, phi_t, df, a_pre, a_post, a_res, bias, iters, bc, n, C,
                                    gy + t0 * N, gr + t0, ghp + t0 * n, ghq + t0 * n,
                                    ghr + t0 * n * n, dfp, dx, ws, num_sms, stream)) !=
            cudaSuccess)
            return e;
        if ((e = cudaEventRecord(rt.computed[s], stream)) != cudaSuccess) return e;

        // outputs of chunk k back to the host
        if ((e = cudaStreamWaitEvent(rt.d2h, rt.computed[s], 0)) != cudaSuccess) return e;
        if ((e = cudaMemcpyAsync(X_next + t0 * K, dx, bc * K * 2, cudaMemcpyDeviceToHost,
                                 rt.d2h)) != cudaSuccess)
            return e;
        if ((e = cudaMemcpyAsync(F_pre + t0 * C, dfp, bc * C * 2, cudaMemcpyDeviceToHost,
                                 rt.d2h)) != cudaSuccess)
            return e;
        if ((e = cudaEventRecord(rt.drained[s], rt.d2h)) != cudaSuccess) return e;
    }
    // the small outputs of the whole batch, behind the last chunk's forward
    // (the d2h stream has waited on every chunk's forward by now)
    const struct {
        void *dst;
        const void *src;
        size_t bytes;
    } small[] = {
        {Y, gy, static_cast<size_t>(B * N * 4)},
        {r, gr, static_cast<size_t>(B * 4)},
        {H_pre, ghp, static_cast<size_t>(B * n * 4)},
        {H_post, ghq, static_cast<size_t>(B * n * 4)},
        {H_res, ghr, static_cast<size_t>(B * n * n * 4)},
    };
    for (const auto &o : small)
        if ((e = cudaMemcpyAsync(o.dst, o.src, o.bytes, cudaMemcpyDeviceToHost, rt.d2h)) !=
            cudaSuccess)
            return e;
    const int last = static_cast<int>((chunks - 1) % kSlots);
    if ((e = cudaEventRecord(rt.drained[last], rt.d2h)) != cudaSuccess) return e;
    // the caller's stream continues once every output is on the host
    for (int s = 0; s < kSlots && s < chunks; ++s)
        if ((e = cudaStreamWaitEvent(stream, rt.drained[s], 0)) != cudaSuccess) return e;
    return cudaSuccess;
}

}  // namespace mhc

extern "C" int mhc_testing_host_chunks(int64_t B, int64_t *sizes, int64_t capacity,
                                       int64_t *count)
{
    if (B < 0 || count == nullptr || capacity < 0 || (capacity > 0 && sizes == nullptr))
        return MHC_ERR_INVALID;
    const std::vector<int64_t> plan =
        mhc::chunk_sizes(B, B < mhc::kHostChunkTokens ? B : mhc::kHostChunkTokens);
    *count = static_cast<int64_t>(plan.size());
    for (int64_t i = 0; i < *count && i < capacity; ++i) sizes[i] = plan[i];
    return MHC_OK;
}
