// C ABI of the mHC forward library (declared in include/mhc.h): argument
// validation on the host, then the kernels of gemm_rms.cu, coeffs.cu,
// apply.cu and decode_pre.cu on the caller's stream.  No exception crosses this boundary and
// nothing here allocates device memory.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "check.cuh"
#include "mhc.h"
#include "mhc_internal.h"
#include "mhc_testing.h"

namespace mhc {

// Readers of the per-file device check records (empty in the default build).
namespace {
std::mutex g_check_mu;
CheckReader g_check_readers[16];
int g_check_count = 0;
}  // namespace

bool register_check_reader(CheckReader reader)
{
    std::lock_guard<std::mutex> lock(g_check_mu);
    if (g_check_count < 16) g_check_readers[g_check_count++] = reader;
    return true;
}

// The first failing record that mhc_device_status reported, kept until
// mhc_testing_check_record reads it.
std::mutex g_check_status_mu;
CheckRecord g_last_check{};

// Reads and clears every record; the first failing one goes to *first.
cudaError_t read_and_clear_checks(CheckRecord *first)
{
    *first = CheckRecord{};
    std::lock_guard<std::mutex> lock(g_check_mu);
    for (int i = 0; i < g_check_count; ++i) {
        CheckRecord rec{};
        const cudaError_t e = g_check_readers[i](&rec);
        if (e != cudaSuccess) return e;
        if (rec.status != 0 && first->status == 0) *first = rec;
    }
    return cudaSuccess;
}

#ifdef MHC_CHECK
namespace {
__global__ void check_selftest_kernel(float *buf)
{
    constexpr int64_t kExtent = 16;
    if (in_range(900, kExtent, 1, kExtent)) buf[kExtent] = 1.0f;  // refused: never stored
}
}  // namespace
#endif

cudaError_t current_device_info(DeviceInfo *info)
{
    constexpr int kMaxDevices = 64;
    static DeviceInfo cache[kMaxDevices];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) {
        std::lock_guard<std::mutex> lock(mu);
        if (cache[dev].device == dev) {
            *info = cache[dev];
            return cudaSuccess;
        }
    }
    DeviceInfo d;
    d.device = dev;
    if ((e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    if ((e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) !=
        cudaSuccess)
        return e;
    if ((e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) !=
        cudaSuccess)
        return e;
    if (dev >= 0 && dev < kMaxDevices) {
        std::lock_guard<std::mutex> lock(mu);
        cache[dev] = d;
    }
    *info = d;
    return cudaSuccess;
}

namespace {

struct Buf {
    const void *p;
    size_t bytes;
};

bool overlaps(const Buf &a, const Buf &b)
{
    if (a.bytes == 0 || b.bytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape rules shared by every call.  Returns MHC_OK or the error.
int check_shape(int64_t B, int n, int64_t C, bool needs_c)
{
    if (B < 0) return MHC_ERR_INVALID;
    if (n < 1 || n > 8) return MHC_ERR_UNSUPPORTED;
    if (needs_c) {
        if (C < 8 || C % 8 != 0) return MHC_ERR_UNSUPPORTED;
        // K = n*C is addressed with 32-bit TMA coordinates and int kernel arguments
        if (static_cast<int64_t>(n) * C > (int64_t{1} << 30)) return MHC_ERR_UNSUPPORTED;
    }
    // token rows are TMA coordinates, 32-bit signed
    if (B >= (int64_t{1} << 31)) return MHC_ERR_UNSUPPORTED;
    return MHC_OK;
}

int check_ptrs(const Buf *bufs, int count)
{
    for (int i = 0; i < count; ++i)
        if (bufs[i].p == nullptr) return MHC_ERR_INVALID;
    for (int i = 0; i < count; ++i)
        if (!aligned16(bufs[i].p)) return MHC_ERR_ALIGN;
    return MHC_OK;
}

// Outputs must not overlap inputs or each other.  `alias_ok` names one
// (output, input) pair that may be exactly equal.
int check_overlap(const Buf *outs, int n_out, const Buf *ins, int n_in, const void *alias_out,
                  const void *alias_in)
{
    for (int i = 0; i < n_out; ++i) {
        for (int j = 0; j < n_in; ++j) {
            if (outs[i].p == alias_out && ins[j].p == alias_in && alias_out == alias_in &&
                outs[i].bytes == ins[j].bytes)
                continue;
            if (overlaps(outs[i], ins[j])) return MHC_ERR_INVALID;
        }
        for (int j = i + 1; j < n_out; ++j)
            if (overlaps(outs[i], outs[j])) return MHC_ERR_INVALID;
    }
    return MHC_OK;
}

// Whether the pointer checks of the device-memory entry points run (on unless a
// test turns them off to time their cost).
std::atomic<int> g_memory_checks{1};

// Every buffer must be device memory of the current device (cudaMalloc,
// stream-ordered pools or mapped VMM ranges): a host pointer, managed memory
// or another GPU's memory reached over peer access is MHC_ERR_INVALID, before
// anything is launched.  The kernels' TMA descriptors and stores assume local
// device memory.
int check_on_device(const Buf *bufs, int count, const DeviceInfo &info)
{
    if (!g_memory_checks.load(std::memory_order_relaxed)) return MHC_OK;
    for (int i = 0; i < count; ++i) {
        cudaPointerAttributes a{};
        if (cudaPointerGetAttributes(&a, bufs[i].p) != cudaSuccess) {
            cudaGetLastError();  // not sticky; clear it
            return MHC_ERR_INVALID;
        }
        if (a.type != cudaMemoryTypeDevice || a.device != info.device) return MHC_ERR_INVALID;
    }
    return MHC_OK;
}

// Every buffer must be host memory (page-locked or pageable), as the runtime
// records it: device or managed memory is MHC_ERR_INVALID.
int check_on_host(const Buf *bufs, int count)
{
    for (int i = 0; i < count; ++i) {
        cudaPointerAttributes a{};
        if (cudaPointerGetAttributes(&a, bufs[i].p) != cudaSuccess) {
            cudaGetLastError();  // not sticky; clear it
            return MHC_ERR_INVALID;
        }
        if (a.type != cudaMemoryTypeHost && a.type != cudaMemoryTypeUnregistered)
            return MHC_ERR_INVALID;
    }
    return MHC_OK;
}

int check_device(DeviceInfo *info)
{
    if (current_device_info(info) != cudaSuccess) return MHC_ERR_CUDA;
    if (info->cc_major != 10 || info->cc_minor != 3) return MHC_ERR_UNSUPPORTED;
    return MHC_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MHC_OK : MHC_ERR_CUDA; }

size_t bf16_bytes(int64_t count) { return static_cast<size_t>(count) * 2; }
size_t f32_bytes(int64_t count) { return static_cast<size_t>(count) * 4; }

#define MHC_TRY(expr)                   \
    do {                                \
        const int st_ = (expr);         \
        if (st_ != MHC_OK) return st_;  \
    } while (0)

// Batches up to this size take the one-launch steps 1-4a kernel.  Measured on
// GB300 against the kernel chain (µs per forward in a CUDA graph): 1.6-2.7x
// faster up to 512 tokens (the chain is bound by launch and reduction latency
// there), 17-43% faster at 1024 (n = 4, C = 7168 and n = 8, C = 4096), within
// 2% at 2048; from 2560 the chain is as fast or faster (3-4% at 3072).
constexpr int64_t kDecodeMaxTokens = 2048;

// Up to this batch the one-launch kernel also forms X_next (step 4b) from the
// coefficients it holds; above it a kernel of its own does, with more loads in
// flight per SM than the one-launch kernel's ten warps.
constexpr int64_t kDecodeXnextMaxTokens = 256;

// mhc_forward's own choice (and that of its fp32-weight form): the one-launch
// steps 1-4a kernel up to kDecodeMaxTokens, else the kernel chain.
bool takes_decode_path(int64_t B, int n, int64_t C)
{
    return B <= kDecodeMaxTokens && decode_pre_eligible(B, n, C);
}

enum class Path {
    Auto,           // decode_pre for small batches, else the kernel chain
    Chain,          // gemm_rms, coeffs, pre_apply
    Fused,          // fused_pre (test hook)
    Decode,         // decode_pre (test hook for any eligible batch)
    DecodeStalled,  // decode_pre whose grid barrier never completes (test hook)
};

}  // namespace

size_t forward_workspace_bytes(int64_t B, int n, int64_t C, int num_sms)
{
    size_t w = gemm_rms_workspace_bytes(B, n, C, num_sms);
    const size_t f = fused_pre_workspace_bytes(B, n, C, num_sms);
    const size_t d = decode_pre_workspace_bytes(B, n, C, num_sms);
    if (f > w) w = f;
    if (d > w) w = d;
    return w;
}

// The coefficient arguments of the GEMM's finalize (steps 2 and 3).
static CoefArgs coef_args(float a_pre, float a_post, float a_res, const float *bias, int iters,
                          int n, float *H_pre, float *H_post, float *H_res)
{
    CoefArgs c;
    c.bias = bias;
    c.a_pre = a_pre;
    c.a_post = a_post;
    c.a_res = a_res;
    c.iters = iters;
    c.n = n;
    c.H_pre = H_pre;
    c.H_post = H_post;
    c.H_res = H_res;
    return c;
}

// The kernels of one forward for a path (arguments already valid and the path
// eligible): steps 1-4a by the path, then the X_next kernel.
static cudaError_t launch_forward(const uint16_t *X, const uint16_t *phi_t, const uint16_t *F_out,
                                  float a_pre, float a_post, float a_res, const float *bias,
                                  int iters, int64_t B, int n, int64_t C, float *Y, float *r,
                                  float *H_pre, float *H_post, float *H_res, uint16_t *F_pre,
                                  uint16_t *X_next, void *workspace, int num_sms, cudaStream_t s,
                                  Path path, uint64_t wait_limit_ns)
{
    if (path == Path::Auto) path = takes_decode_path(B, n, C) ? Path::Decode : Path::Chain;
    cudaError_t e;
    if (path == Path::Fused) {
        // steps 1-4a in one kernel that reads X from HBM once
        e = launch_fused_pre(X, phi_t, a_pre, a_post, a_res, bias, iters, B, n, C, Y, r, H_pre,
                             H_post, H_res, F_pre, workspace, num_sms, s);
    } else if (path == Path::Decode || path == Path::DecodeStalled) {
        // steps 1-4a in one launch, and 4b with them for the smallest batches
        const bool with_4b = B <= kDecodeXnextMaxTokens;
        e = launch_decode_pre(X, phi_t, a_pre, a_post, a_res, bias, iters, B, n, C, Y, r, H_pre,
                              H_post, H_res, F_pre, F_out, with_4b ? X_next : nullptr, workspace,
                              num_sms, s, wait_limit_ns, path == Path::DecodeStalled ? 1 : 0);
        if (with_4b) return e;
    } else {
        // steps 1-3: the GEMM's finalize forms the coefficients of each finished token
        e = launch_gemm_rms(X, phi_t, B, n, C, Y, r, workspace, num_sms, s, kWaitLimitNs, -1,
                            coef_args(a_pre, a_post, a_res, bias, iters, n, H_pre, H_post, H_res));
        if (e == cudaSuccess) e = launch_pre_apply(X, H_pre, B, n, C, F_pre, s);
    }
    if (e == cudaSuccess) e = launch_post_res_apply(X, F_out, H_res, H_post, B, n, C, X_next, s);
    return e;
}

cudaError_t run_forward_device(const uint16_t *X, const uint16_t *phi_t, const uint16_t *F_out,
                               float a_pre, float a_post, float a_res, const float *bias,
                               int iters, int64_t B, int n, int64_t C, float *Y, float *r,
                               float *H_pre, float *H_post, float *H_res, uint16_t *F_pre,
                               uint16_t *X_next, void *workspace, int num_sms,
                               cudaStream_t stream)
{
    return launch_forward(X, phi_t, F_out, a_pre, a_post, a_res, bias, iters, B, n, C, Y, r,
                          H_pre, H_post, H_res, F_pre, X_next, workspace, num_sms, stream,
                          Path::Auto, kWaitLimitNs);
}

}  // namespace mhc

using namespace mhc;

static int forward_checked(const mhc_bf16 *X, const mhc_bf16 *phi_t, const mhc_bf16 *F_out,
                           float alpha_pre, float alpha_post, float alpha_res, const float *bias,
                           int iters, int64_t B, int n, int64_t C, float *Y, float *r,
                           float *H_pre, float *H_post, float *H_res, mhc_bf16 *F_pre,
                           mhc_bf16 *X_next, void *workspace, size_t workspace_bytes,
                           mhc_stream_t stream, Path path, uint64_t wait_limit_ns = kWaitLimitNs)
{
    MHC_TRY(check_shape(B, n, C, true));
    if (iters < 0) return MHC_ERR_INVALID;
    if (B == 0) return MHC_OK;
    const int N = num_coeffs(n);
    const int64_t K = n * C;
    const Buf ins[] = {{X, bf16_bytes(B * K)}, {phi_t, bf16_bytes(int64_t{N} * K)},
                       {F_out, bf16_bytes(B * C)}, {bias, f32_bytes(N)}};
    Buf outs[] = {{Y, f32_bytes(B * N)},        {r, f32_bytes(B)},
                  {H_pre, f32_bytes(B * n)},     {H_post, f32_bytes(B * n)},
                  {H_res, f32_bytes(B * n * n)}, {F_pre, bf16_bytes(B * C)},
                  {X_next, bf16_bytes(B * K)},   {workspace, workspace_bytes}};
    MHC_TRY(check_ptrs(ins, 4));
    MHC_TRY(check_ptrs(outs, 7));
    MHC_TRY(check_overlap(outs, 7, ins, 4, X_next, X));
    DeviceInfo info;
    MHC_TRY(check_device(&info));
    MHC_TRY(check_on_device(ins, 4, info));
    MHC_TRY(check_on_device(outs, 7, info));
    const size_t need = forward_workspace_bytes(B, n, C, info.num_sms);
    if (workspace == nullptr || workspace_bytes < need) return MHC_ERR_WORKSPACE;
    outs[7].bytes = need;
    MHC_TRY(check_ptrs(outs + 7, 1));
    MHC_TRY(check_overlap(outs, 8, ins, 4, X_next, X));
    MHC_TRY(check_on_device(outs + 7, 1, info));
    if (path == Path::Fused && !fused_pre_eligible(B, n, C, info.num_sms))
        return MHC_ERR_UNSUPPORTED;
    if ((path == Path::Decode || path == Path::DecodeStalled) && !decode_pre_eligible(B, n, C))
        return MHC_ERR_UNSUPPORTED;
    return cuda_status(launch_forward(X, phi_t, F_out, alpha_pre, alpha_post, alpha_res, bias,
                                      iters, B, n, C, Y, r, H_pre, H_post, H_res, F_pre, X_next,
                                      workspace, info.num_sms,
                                      reinterpret_cast<cudaStream_t>(stream), path,
                                      wait_limit_ns));
}

static int gemm_rms_checked(const mhc_bf16 *X, const mhc_bf16 *phi_t, int64_t B, int n, int64_t C,
                            float *Y, float *r, void *workspace, size_t workspace_bytes,
                            mhc_stream_t stream, uint64_t wait_limit_ns, int64_t stall_stage)
{
    MHC_TRY(check_shape(B, n, C, true));
    if (B == 0) return MHC_OK;
    const int N = num_coeffs(n);
    const int64_t K = n * C;
    const Buf ins[] = {{X, bf16_bytes(B * K)}, {phi_t, bf16_bytes(int64_t{N} * K)}};
    Buf outs[] = {{Y, f32_bytes(B * N)}, {r, f32_bytes(B)}, {workspace, workspace_bytes}};
    MHC_TRY(check_ptrs(ins, 2));
    MHC_TRY(check_ptrs(outs, 2));
    MHC_TRY(check_overlap(outs, 2, ins, 2, nullptr, nullptr));
    DeviceInfo info;
    MHC_TRY(check_device(&info));
    MHC_TRY(check_on_device(ins, 2, info));
    MHC_TRY(check_on_device(outs, 2, info));
    const size_t need = gemm_rms_workspace_bytes(B, n, C, info.num_sms);
    if (workspace == nullptr || workspace_bytes < need) return MHC_ERR_WORKSPACE;
    outs[2].bytes = need;
    MHC_TRY(check_ptrs(outs + 2, 1));
    MHC_TRY(check_overlap(outs, 3, ins, 2, nullptr, nullptr));
    MHC_TRY(check_on_device(outs + 2, 1, info));
    return cuda_status(launch_gemm_rms(X, phi_t, B, n, C, Y, r, workspace, info.num_sms,
                                       reinterpret_cast<cudaStream_t>(stream), wait_limit_ns,
                                       stall_stage));
}

extern "C" {

const char *mhc_status_str(int status)
{
    switch (status) {
    case MHC_OK: return "MHC_OK";
    case MHC_ERR_INVALID: return "MHC_ERR_INVALID: bad size, NULL pointer, overlap or iters < 0";
    case MHC_ERR_UNSUPPORTED: return "MHC_ERR_UNSUPPORTED: n, C or device not supported";
    case MHC_ERR_ALIGN: return "MHC_ERR_ALIGN: pointer not 16-byte aligned";
    case MHC_ERR_CUDA: return "MHC_ERR_CUDA: CUDA runtime call or launch failed";
    case MHC_ERR_TIMEOUT: return "MHC_ERR_TIMEOUT: a bounded device wait ran out";
    case MHC_ERR_WORKSPACE: return "MHC_ERR_WORKSPACE: workspace missing or too small";
    case MHC_ERR_BOUNDS: return "MHC_ERR_BOUNDS: a device index check failed (MHC_CHECK build)";
    default: return "unknown mhc status";
    }
}

size_t mhc_workspace_bytes(int64_t B, int n, int64_t C)
{
    if (check_shape(B, n, C, true) != MHC_OK) return 0;
    DeviceInfo info;
    if (current_device_info(&info) != cudaSuccess) return 0;
    return forward_workspace_bytes(B, n, C, info.num_sms);
}

int mhc_gemm_rms(const mhc_bf16 *X, const mhc_bf16 *phi_t, int64_t B, int n, int64_t C, float *Y,
                 float *r, void *workspace, size_t workspace_bytes, mhc_stream_t stream)
{
    return gemm_rms_checked(X, phi_t, B, n, C, Y, r, workspace, workspace_bytes, stream,
                            kWaitLimitNs, -1);
}

int mhc_testing_gemm_rms_stalled(const mhc_bf16 *X, const mhc_bf16 *phi_t, int64_t B, int n,
                                 int64_t C, float *Y, float *r, void *workspace,
                                 size_t workspace_bytes, int64_t stall_stage,
                                 uint64_t wait_limit_ns, mhc_stream_t stream)
{
    const uint64_t lo = 1000000ull;
    const uint64_t limit = wait_limit_ns < lo ? lo : (wait_limit_ns > kWaitLimitNs ? kWaitLimitNs
                                                                                   : wait_limit_ns);
    return gemm_rms_checked(X, phi_t, B, n, C, Y, r, workspace, workspace_bytes, stream, limit,
                            stall_stage);
}

int mhc_coeffs(const float *Y, const float *r, float alpha_pre, float alpha_post, float alpha_res,
               const float *bias, int iters, int64_t B, int n, float *H_pre, float *H_post,
               float *H_res, mhc_stream_t stream)
{
    MHC_TRY(check_shape(B, n, 8, false));
    if (iters < 0) return MHC_ERR_INVALID;
    if (B == 0) return MHC_OK;
    const int N = num_coeffs(n);
    const Buf ins[] = {{Y, f32_bytes(B * N)}, {r, f32_bytes(B)}, {bias, f32_bytes(N)}};
    const Buf outs[] = {{H_pre, f32_bytes(B * n)}, {H_post, f32_bytes(B * n)},
                        {H_res, f32_bytes(B * n * n)}};
    MHC_TRY(check_ptrs(ins, 3));
    MHC_TRY(check_ptrs(outs, 3));
    MHC_TRY(check_overlap(outs, 3, ins, 3, nullptr, nullptr));
    DeviceInfo info;
    MHC_TRY(check_device(&info));
    MHC_TRY(check_on_device(ins, 3, info));
    MHC_TRY(check_on_device(outs, 3, info));
    return cuda_status(launch_coeffs(Y, r, alpha_pre, alpha_post, alpha_res, bias, iters, B, n,
                                     H_pre, H_post, H_res, reinterpret_cast<cudaStream_t>(stream)));
}

int mhc_gemm_rms_coeffs(const mhc_bf16 *X, const mhc_bf16 *phi_t, float alpha_pre,
                        float alpha_post, float alpha_res, const float *bias, int iters,
                        int64_t B, int n, int64_t C, float *Y, float *r, float *H_pre,
                        float *H_post, float *H_res, void *workspace, size_t workspace_bytes,
                        mhc_stream_t stream)
{
    MHC_TRY(check_shape(B, n, C, true));
    if (iters < 0) return MHC_ERR_INVALID;
    if (B == 0) return MHC_OK;
    const int N = num_coeffs(n);
    const int64_t K = n * C;
    const Buf ins[] = {{X, bf16_bytes(B * K)}, {phi_t, bf16_bytes(int64_t{N} * K)},
                       {bias, f32_bytes(N)}};
    Buf outs[] = {{Y, f32_bytes(B * N)},         {r, f32_bytes(B)},
                  {H_pre, f32_bytes(B * n)},     {H_post, f32_bytes(B * n)},
                  {H_res, f32_bytes(B * n * n)}, {workspace, workspace_bytes}};
    MHC_TRY(check_ptrs(ins, 3));
    MHC_TRY(check_ptrs(outs, 5));
    MHC_TRY(check_overlap(outs, 5, ins, 3, nullptr, nullptr));
    DeviceInfo info;
    MHC_TRY(check_device(&info));
    MHC_TRY(check_on_device(ins, 3, info));
    MHC_TRY(check_on_device(outs, 5, info));
    const size_t need = gemm_rms_workspace_bytes(B, n, C, info.num_sms);
    if (workspace == nullptr || workspace_bytes < need) return MHC_ERR_WORKSPACE;
    outs[5].bytes = need;
    MHC_TRY(check_ptrs(outs + 5, 1));
    MHC_TRY(check_overlap(outs, 6, ins, 3, nullptr, nullptr));
    MHC_TRY(check_on_device(outs + 5, 1, info));
    return cuda_status(launch_gemm_rms(
        X, phi_t, B, n, C, Y, r, workspace, info.num_sms, reinterpret_cast<cudaStream_t>(stream),
        kWaitLimitNs, -1,
        coef_args(alpha_pre, alpha_post, alpha_res, bias, iters, n, H_pre, H_post, H_res)));
}

int mhc_pre_apply(const mhc_bf16 *X, const float *H_pre, int64_t B, int n, int64_t C,
                  mhc_bf16 *F_pre, mhc_stream_t stream)
{
    MHC_TRY(check_shape(B, n, C, true));
    if (B == 0) return MHC_OK;
    const Buf ins[] = {{X, bf16_bytes(B * n * C)}, {H_pre, f32_bytes(B * n)}};
    const Buf outs[] = {{F_pre, bf16_bytes(B * C)}};
    MHC_TRY(check_ptrs(ins, 2));
    MHC_TRY(check_ptrs(outs, 1));
    MHC_TRY(check_overlap(outs, 1, ins, 2, nullptr, nullptr));
    DeviceInfo info;
    MHC_TRY(check_device(&info));
    MHC_TRY(check_on_device(ins, 2, info));
    MHC_TRY(check_on_device(outs, 1, info));
    return cuda_status(
        launch_pre_apply(X, H_pre, B, n, C, F_pre, reinterpret_cast<cudaStream_t>(stream)));
}

int mhc_post_res_apply(const mhc_bf16 *X, const mhc_bf16 *F_out, const float *H_res,
                       const float *H_post, int64_t B, int n, int64_t C, mhc_bf16 *X_next,
                       mhc_stream_t stream)
{
    MHC_TRY(check_shape(B, n, C, true));
    if (B == 0) return MHC_OK;
    const Buf ins[] = {{X, bf16_bytes(B * n * C)}, {F_out, bf16_bytes(B * C)},
                       {H_res, f32_bytes(B * n * n)}, {H_post, f32_bytes(B * n)}};
    const Buf outs[] = {{X_next, bf16_bytes(B * n * C)}};
    MHC_TRY(check_ptrs(ins, 4));
    MHC_TRY(check_ptrs(outs, 1));
    MHC_TRY(check_overlap(outs, 1, ins, 4, X_next, X));
    DeviceInfo info;
    MHC_TRY(check_device(&info));
    MHC_TRY(check_on_device(ins, 4, info));
    MHC_TRY(check_on_device(outs, 1, info));
    return cuda_status(launch_post_res_apply(X, F_out, H_res, H_post, B, n, C, X_next,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

int mhc_forward(const mhc_bf16 *X, const mhc_bf16 *phi_t, const mhc_bf16 *F_out, float alpha_pre,
                float alpha_post, float alpha_res, const float *bias, int iters, int64_t B, int n,
                int64_t C, float *Y, float *r, float *H_pre, float *H_post, float *H_res,
                mhc_bf16 *F_pre, mhc_bf16 *X_next, void *workspace, size_t workspace_bytes,
                mhc_stream_t stream)
{
    return forward_checked(X, phi_t, F_out, alpha_pre, alpha_post, alpha_res, bias, iters, B, n,
                           C, Y, r, H_pre, H_post, H_res, F_pre, X_next, workspace,
                           workspace_bytes, stream, Path::Auto);
}

#define MHC_FORWARD_ARGS                                                                         \
    const mhc_bf16 *X, const mhc_bf16 *phi_t, const mhc_bf16 *F_out, float alpha_pre,            \
        float alpha_post, float alpha_res, const float *bias, int iters, int64_t B, int n,       \
        int64_t C, float *Y, float *r, float *H_pre, float *H_post, float *H_res,                \
        mhc_bf16 *F_pre, mhc_bf16 *X_next, void *workspace, size_t workspace_bytes,              \
        mhc_stream_t stream
#define MHC_FORWARD_PASS                                                                         \
    X, phi_t, F_out, alpha_pre, alpha_post, alpha_res, bias, iters, B, n, C, Y, r, H_pre,        \
        H_post, H_res, F_pre, X_next, workspace, workspace_bytes, stream

int mhc_testing_forward_fused(MHC_FORWARD_ARGS)
{
    return forward_checked(MHC_FORWARD_PASS, Path::Fused);
}

int mhc_testing_forward_chain(MHC_FORWARD_ARGS)
{
    return forward_checked(MHC_FORWARD_PASS, Path::Chain);
}

int mhc_testing_forward_decode(MHC_FORWARD_ARGS)
{
    return forward_checked(MHC_FORWARD_PASS, Path::Decode);
}

int mhc_testing_forward_decode_stalled(MHC_FORWARD_ARGS, uint64_t wait_limit_ns)
{
    uint64_t lim = wait_limit_ns;
    if (lim < 1000000ull) lim = 1000000ull;
    if (lim > kWaitLimitNs) lim = kWaitLimitNs;
    return forward_checked(MHC_FORWARD_PASS, Path::DecodeStalled, lim);
}

#undef MHC_FORWARD_ARGS
#undef MHC_FORWARD_PASS

int mhc_testing_recip(const float *in, float *out, int64_t count, mhc_stream_t stream)
{
    if (count < 0) return MHC_ERR_INVALID;
    if (count == 0) return MHC_OK;
    const Buf ins[] = {{in, f32_bytes(count)}};
    const Buf outs[] = {{out, f32_bytes(count)}};
    MHC_TRY(check_ptrs(ins, 1));
    MHC_TRY(check_ptrs(outs, 1));
    MHC_TRY(check_overlap(outs, 1, ins, 1, nullptr, nullptr));
    DeviceInfo info;
    MHC_TRY(check_device(&info));
    MHC_TRY(check_on_device(ins, 1, info));
    MHC_TRY(check_on_device(outs, 1, info));
    return cuda_status(launch_recip(in, out, count, reinterpret_cast<cudaStream_t>(stream)));
}

// ---------------------------------------- fp32-weight precision variant

int mhc_split_phi(const float *phi_t, int n, int64_t C, mhc_bf16 *phi_split, mhc_stream_t stream)
{
    MHC_TRY(check_shape(1, n, C, true));
    const int N = num_coeffs(n);
    const int64_t K = n * C;
    const Buf ins[] = {{phi_t, f32_bytes(int64_t{N} * K)}};
    const Buf outs[] = {{phi_split, bf16_bytes(int64_t{2} * N * K)}};
    MHC_TRY(check_ptrs(ins, 1));
    MHC_TRY(check_ptrs(outs, 1));
    MHC_TRY(check_overlap(outs, 1, ins, 1, nullptr, nullptr));
    DeviceInfo info;
    MHC_TRY(check_device(&info));
    MHC_TRY(check_on_device(ins, 1, info));
    MHC_TRY(check_on_device(outs, 1, info));
    return cuda_status(launch_split_phi(phi_t, n, C, phi_split,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

int mhc_gemm_rms_split(const mhc_bf16 *X, const mhc_bf16 *phi_split, int64_t B, int n, int64_t C,
                       float *Y, float *r, void *workspace, size_t workspace_bytes,
                       mhc_stream_t stream)
{
    MHC_TRY(check_shape(B, n, C, true));
    if (B == 0) return MHC_OK;
    const int N = num_coeffs(n);
    const int64_t K = n * C;
    const Buf ins[] = {{X, bf16_bytes(B * K)}, {phi_split, bf16_bytes(int64_t{2} * N * K)}};
    Buf outs[] = {{Y, f32_bytes(B * N)}, {r, f32_bytes(B)}, {workspace, workspace_bytes}};
    MHC_TRY(check_ptrs(ins, 2));
    MHC_TRY(check_ptrs(outs, 2));
    MHC_TRY(check_overlap(outs, 2, ins, 2, nullptr, nullptr));
    DeviceInfo info;
    MHC_TRY(check_device(&info));
    MHC_TRY(check_on_device(ins, 2, info));
    MHC_TRY(check_on_device(outs, 2, info));
    const size_t need = gemm_rms_workspace_bytes(B, n, C, info.num_sms);
    if (workspace == nullptr || workspace_bytes < need) return MHC_ERR_WORKSPACE;
    outs[2].bytes = need;
    MHC_TRY(check_ptrs(outs + 2, 1));
    MHC_TRY(check_overlap(outs, 3, ins, 2, nullptr, nullptr));
    MHC_TRY(check_on_device(outs + 2, 1, info));
    return cuda_status(launch_gemm_rms_split(X, phi_split, B, n, C, Y, r, workspace, info.num_sms,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

int mhc_post_res_apply_f32(const mhc_bf16 *X, const float *F_out, const float *H_res,
                           const float *H_post, int64_t B, int n, int64_t C, mhc_bf16 *X_next,
                           mhc_stream_t stream)
{
    MHC_TRY(check_shape(B, n, C, true));
    if (B == 0) return MHC_OK;
    const int64_t K = n * C;
    const Buf ins[] = {{X, bf16_bytes(B * K)}, {F_out, f32_bytes(B * C)},
                       {H_res, f32_bytes(B * n * n)}, {H_post, f32_bytes(B * n)}};
    const Buf outs[] = {{X_next, bf16_bytes(B * K)}};
    MHC_TRY(check_ptrs(ins, 4));
    MHC_TRY(check_ptrs(outs, 1));
    MHC_TRY(check_overlap(outs, 1, ins, 4, X_next, X));
    DeviceInfo info;
    MHC_TRY(check_device(&info));
    MHC_TRY(check_on_device(ins, 4, info));
    MHC_TRY(check_on_device(outs, 1, info));
    return cuda_status(launch_post_res_apply_f32(X, F_out, H_res, H_post, B, n, C, X_next,
                                                 reinterpret_cast<cudaStream_t>(stream)));
}

int mhc_forward_f32w(const mhc_bf16 *X, const mhc_bf16 *phi_split, const float *F_out,
                     float alpha_pre, float alpha_post, float alpha_res, const float *bias,
                     int iters, int64_t B, int n, int64_t C, float *Y, float *r, float *H_pre,
                     float *H_post, float *H_res, mhc_bf16 *F_pre, mhc_bf16 *X_next,
                     void *workspace, size_t workspace_bytes, mhc_stream_t stream)
{
    MHC_TRY(check_shape(B, n, C, true));
    if (iters < 0) return MHC_ERR_INVALID;
    if (B == 0) return MHC_OK;
    const int N = num_coeffs(n);
    const int64_t K = n * C;
    const Buf ins[] = {{X, bf16_bytes(B * K)}, {phi_split, bf16_bytes(int64_t{2} * N * K)},
                       {F_out, f32_bytes(B * C)}, {bias, f32_bytes(N)}};
    Buf outs[] = {{Y, f32_bytes(B * N)},        {r, f32_bytes(B)},
                  {H_pre, f32_bytes(B * n)},     {H_post, f32_bytes(B * n)},
                  {H_res, f32_bytes(B * n * n)}, {F_pre, bf16_bytes(B * C)},
                  {X_next, bf16_bytes(B * K)},   {workspace, workspace_bytes}};
    MHC_TRY(check_ptrs(ins, 4));
    MHC_TRY(check_ptrs(outs, 7));
    MHC_TRY(check_overlap(outs, 7, ins, 4, X_next, X));
    DeviceInfo info;
    MHC_TRY(check_device(&info));
    MHC_TRY(check_on_device(ins, 4, info));
    MHC_TRY(check_on_device(outs, 7, info));
    const size_t need = forward_workspace_bytes(B, n, C, info.num_sms);
    if (workspace == nullptr || workspace_bytes < need) return MHC_ERR_WORKSPACE;
    outs[7].bytes = need;
    MHC_TRY(check_ptrs(outs + 7, 1));
    MHC_TRY(check_overlap(outs, 8, ins, 4, X_next, X));
    MHC_TRY(check_on_device(outs + 7, 1, info));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    bool with_4b = false;
    if (takes_decode_path(B, n, C)) {
        // steps 1-4a in one launch, and 4b with them for the smallest batches
        with_4b = B <= kDecodeXnextMaxTokens;
        e = launch_decode_pre(X, phi_split, alpha_pre, alpha_post, alpha_res, bias, iters, B, n,
                              C, Y, r, H_pre, H_post, H_res, F_pre, F_out,
                              with_4b ? X_next : nullptr, workspace, info.num_sms, s,
                              kWaitLimitNs, 0, true);
    } else {
        e = launch_gemm_rms_split(X, phi_split, B, n, C, Y, r, workspace, info.num_sms, s,
                                  coef_args(alpha_pre, alpha_post, alpha_res, bias, iters, n,
                                            H_pre, H_post, H_res));
        if (e == cudaSuccess) e = launch_pre_apply(X, H_pre, B, n, C, F_pre, s);
    }
    if (e == cudaSuccess && !with_4b)
        e = launch_post_res_apply_f32(X, F_out, H_res, H_post, B, n, C, X_next, s);
    return cuda_status(e);
}

// -------------------------------------------------- fp8 e4m3 variant

static int check_e4m3_shape(int64_t B, int n, int64_t C)
{
    MHC_TRY(check_shape(B, n, C, true));
    if (C % 16 != 0) return MHC_ERR_UNSUPPORTED;  // 16 channels per 128-bit access
    return MHC_OK;
}

int mhc_gemm_rms_e4m3(const uint8_t *X, const uint8_t *phi_t, int64_t B, int n, int64_t C,
                      float *Y, float *r, void *workspace, size_t workspace_bytes,
                      mhc_stream_t stream)
{
    MHC_TRY(check_e4m3_shape(B, n, C));
    if (B == 0) return MHC_OK;
    const int N = num_coeffs(n);
    const int64_t K = n * C;
    const Buf ins[] = {{X, static_cast<size_t>(B * K)}, {phi_t, static_cast<size_t>(N * K)}};
    Buf outs[] = {{Y, f32_bytes(B * N)}, {r, f32_bytes(B)}, {workspace, workspace_bytes}};
    MHC_TRY(check_ptrs(ins, 2));
    MHC_TRY(check_ptrs(outs, 2));
    MHC_TRY(check_overlap(outs, 2, ins, 2, nullptr, nullptr));
    DeviceInfo info;
    MHC_TRY(check_device(&info));
    MHC_TRY(check_on_device(ins, 2, info));
    MHC_TRY(check_on_device(outs, 2, info));
    const size_t need = gemm_rms_workspace_bytes(B, n, C, info.num_sms);
    if (workspace == nullptr || workspace_bytes < need) return MHC_ERR_WORKSPACE;
    outs[2].bytes = need;
    MHC_TRY(check_ptrs(outs + 2, 1));
    MHC_TRY(check_overlap(outs, 3, ins, 2, nullptr, nullptr));
    MHC_TRY(check_on_device(outs + 2, 1, info));
    return cuda_status(launch_gemm_rms_e4m3(X, phi_t, B, n, C, Y, r, workspace, info.num_sms,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

int mhc_pre_apply_e4m3(const uint8_t *X, const float *H_pre, int64_t B, int n, int64_t C,
                       uint8_t *F_pre, mhc_stream_t stream)
{
    MHC_TRY(check_e4m3_shape(B, n, C));
    if (B == 0) return MHC_OK;
    const int64_t K = n * C;
    const Buf ins[] = {{X, static_cast<size_t>(B * K)}, {H_pre, f32_bytes(B * n)}};
    const Buf outs[] = {{F_pre, static_cast<size_t>(B * C)}};
    MHC_TRY(check_ptrs(ins, 2));
    MHC_TRY(check_ptrs(outs, 1));
    MHC_TRY(check_overlap(outs, 1, ins, 2, nullptr, nullptr));
    DeviceInfo info;
    MHC_TRY(check_device(&info));
    MHC_TRY(check_on_device(ins, 2, info));
    MHC_TRY(check_on_device(outs, 1, info));
    return cuda_status(launch_pre_apply_e4m3(X, H_pre, B, n, C, F_pre,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

int mhc_post_res_apply_e4m3(const uint8_t *X, const uint8_t *F_out, const float *H_res,
                            const float *H_post, int64_t B, int n, int64_t C, uint8_t *X_next,
                            mhc_stream_t stream)
{
    MHC_TRY(check_e4m3_shape(B, n, C));
    if (B == 0) return MHC_OK;
    const int64_t K = n * C;
    const Buf ins[] = {{X, static_cast<size_t>(B * K)}, {F_out, static_cast<size_t>(B * C)},
                       {H_res, f32_bytes(B * n * n)}, {H_post, f32_bytes(B * n)}};
    const Buf outs[] = {{X_next, static_cast<size_t>(B * K)}};
    MHC_TRY(check_ptrs(ins, 4));
    MHC_TRY(check_ptrs(outs, 1));
    MHC_TRY(check_overlap(outs, 1, ins, 4, X_next, X));
    DeviceInfo info;
    MHC_TRY(check_device(&info));
    MHC_TRY(check_on_device(ins, 4, info));
    MHC_TRY(check_on_device(outs, 1, info));
    return cuda_status(launch_post_res_apply_e4m3(X, F_out, H_res, H_post, B, n, C, X_next,
                                                  reinterpret_cast<cudaStream_t>(stream)));
}

int mhc_forward_e4m3(const uint8_t *X, const uint8_t *phi_t, const uint8_t *F_out,
                     float alpha_pre, float alpha_post, float alpha_res, const float *bias,
                     int iters, int64_t B, int n, int64_t C, float *Y, float *r, float *H_pre,
                     float *H_post, float *H_res, uint8_t *F_pre, uint8_t *X_next,
                     void *workspace, size_t workspace_bytes, mhc_stream_t stream)
{
    MHC_TRY(check_e4m3_shape(B, n, C));
    if (iters < 0) return MHC_ERR_INVALID;
    if (B == 0) return MHC_OK;
    const int N = num_coeffs(n);
    const int64_t K = n * C;
    const Buf ins[] = {{X, static_cast<size_t>(B * K)}, {phi_t, static_cast<size_t>(N * K)},
                       {F_out, static_cast<size_t>(B * C)}, {bias, f32_bytes(N)}};
    Buf outs[] = {{Y, f32_bytes(B * N)},        {r, f32_bytes(B)},
                  {H_pre, f32_bytes(B * n)},     {H_post, f32_bytes(B * n)},
                  {H_res, f32_bytes(B * n * n)}, {F_pre, static_cast<size_t>(B * C)},
                  {X_next, static_cast<size_t>(B * K)}, {workspace, workspace_bytes}};
    MHC_TRY(check_ptrs(ins, 4));
    MHC_TRY(check_ptrs(outs, 7));
    MHC_TRY(check_overlap(outs, 7, ins, 4, X_next, X));
    DeviceInfo info;
    MHC_TRY(check_device(&info));
    MHC_TRY(check_on_device(ins, 4, info));
    MHC_TRY(check_on_device(outs, 7, info));
    const size_t need = gemm_rms_workspace_bytes(B, n, C, info.num_sms);
    if (workspace == nullptr || workspace_bytes < need) return MHC_ERR_WORKSPACE;
    outs[7].bytes = need;
    MHC_TRY(check_ptrs(outs + 7, 1));
    MHC_TRY(check_overlap(outs, 8, ins, 4, X_next, X));
    MHC_TRY(check_on_device(outs + 7, 1, info));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = launch_gemm_rms_e4m3(X, phi_t, B, n, C, Y, r, workspace, info.num_sms, s,
                                         coef_args(alpha_pre, alpha_post, alpha_res, bias, iters,
                                                   n, H_pre, H_post, H_res));
    if (e == cudaSuccess) e = launch_pre_apply_e4m3(X, H_pre, B, n, C, F_pre, s);
    if (e == cudaSuccess)
        e = launch_post_res_apply_e4m3(X, F_out, H_res, H_post, B, n, C, X_next, s);
    return cuda_status(e);
}

// Shape rules of mhc_rmsnorm_gemm.
static int check_rng_shape(int64_t M, int64_t K, int64_t N, float eps)
{
    if (M < 0 || !(eps >= 0.0f) || eps > 3.0e38f) return MHC_ERR_INVALID;
    if (K < 8 || K % 8 != 0 || K > (int64_t{1} << 30)) return MHC_ERR_UNSUPPORTED;
    if (N < 8 || N % 8 != 0 || N > (int64_t{1} << 24)) return MHC_ERR_UNSUPPORTED;
    if (M >= (int64_t{1} << 31)) return MHC_ERR_UNSUPPORTED;
    return MHC_OK;
}

size_t mhc_rmsnorm_gemm_workspace_bytes(int64_t M, int64_t K, int64_t N)
{
    if (check_rng_shape(M, K, N, 0.0f) != MHC_OK) return 0;
    DeviceInfo info;
    if (current_device_info(&info) != cudaSuccess) return 0;
    return rmsnorm_gemm_workspace_bytes(M, K, N, info.num_sms);
}

int mhc_rmsnorm_gemm(const mhc_bf16 *A, const mhc_bf16 *B_t, int64_t M, int64_t K, int64_t N,
                     float eps, mhc_bf16 *C, void *workspace, size_t workspace_bytes,
                     mhc_stream_t stream)
{
    MHC_TRY(check_rng_shape(M, K, N, eps));
    if (M == 0) return MHC_OK;
    const Buf ins[] = {{A, bf16_bytes(M * K)}, {B_t, bf16_bytes(N * K)}};
    Buf outs[] = {{C, bf16_bytes(M * N)}, {workspace, workspace_bytes}};
    MHC_TRY(check_ptrs(ins, 2));
    MHC_TRY(check_ptrs(outs, 1));
    MHC_TRY(check_overlap(outs, 1, ins, 2, nullptr, nullptr));
    DeviceInfo info;
    MHC_TRY(check_device(&info));
    MHC_TRY(check_on_device(ins, 2, info));
    MHC_TRY(check_on_device(outs, 1, info));
    const size_t need = rmsnorm_gemm_workspace_bytes(M, K, N, info.num_sms);
    if (need > 0) {
        if (workspace == nullptr || workspace_bytes < need) return MHC_ERR_WORKSPACE;
        outs[1].bytes = need;
        MHC_TRY(check_ptrs(outs + 1, 1));
        MHC_TRY(check_overlap(outs, 2, ins, 2, nullptr, nullptr));
        MHC_TRY(check_on_device(outs + 1, 1, info));
    }
    return cuda_status(launch_rmsnorm_gemm(A, B_t, M, K, N, eps, C, need > 0 ? workspace : nullptr,
                                           info.num_sms, reinterpret_cast<cudaStream_t>(stream)));
}

size_t mhc_forward_host_scratch_bytes(int64_t B, int n, int64_t C)
{
    if (check_shape(B, n, C, true) != MHC_OK || B == 0) return 0;
    DeviceInfo info;
    if (current_device_info(&info) != cudaSuccess) return 0;
    return host_chunk_layout(B, n, C, info.num_sms).total;
}

int mhc_forward_host(const mhc_bf16 *X, const mhc_bf16 *phi_t, const mhc_bf16 *F_out,
                     float alpha_pre, float alpha_post, float alpha_res, const float *bias,
                     int iters, int64_t B, int n, int64_t C, float *Y, float *r, float *H_pre,
                     float *H_post, float *H_res, mhc_bf16 *F_pre, mhc_bf16 *X_next,
                     void *scratch, size_t scratch_bytes, mhc_stream_t stream)
{
    MHC_TRY(check_shape(B, n, C, true));
    if (iters < 0) return MHC_ERR_INVALID;
    if (B == 0) return MHC_OK;
    const int N = num_coeffs(n);
    const int64_t K = n * C;
    const Buf host_in[] = {{X, bf16_bytes(B * K)}, {F_out, bf16_bytes(B * C)}};
    const Buf dev_in[] = {{phi_t, bf16_bytes(int64_t{N} * K)}, {bias, f32_bytes(N)}};
    Buf outs[] = {{Y, f32_bytes(B * N)},        {r, f32_bytes(B)},
                  {H_pre, f32_bytes(B * n)},     {H_post, f32_bytes(B * n)},
                  {H_res, f32_bytes(B * n * n)}, {F_pre, bf16_bytes(B * C)},
                  {X_next, bf16_bytes(B * K)},   {scratch, scratch_bytes}};
    const Buf ins[] = {host_in[0], host_in[1], dev_in[0], dev_in[1]};
    MHC_TRY(check_ptrs(ins, 4));
    MHC_TRY(check_ptrs(outs, 8));
    MHC_TRY(check_overlap(outs, 8, ins, 4, X_next, X));
    DeviceInfo info;
    MHC_TRY(check_device(&info));
    MHC_TRY(check_on_host(host_in, 2));
    MHC_TRY(check_on_host(outs, 7));
    MHC_TRY(check_on_device(dev_in, 2, info));
    MHC_TRY(check_on_device(outs + 7, 1, info));
    if (scratch_bytes < host_chunk_layout(B, n, C, info.num_sms).total) return MHC_ERR_WORKSPACE;
    return cuda_status(run_forward_host(X, phi_t, F_out, alpha_pre, alpha_post, alpha_res, bias,
                                        iters, B, n, C, Y, r, H_pre, H_post, H_res, F_pre,
                                        X_next, scratch, info.num_sms,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

int mhc_testing_memory_checks(int on)
{
    return g_memory_checks.exchange(on != 0 ? 1 : 0);
}

int mhc_testing_check_build(void) { return kCheckBuild ? 1 : 0; }

int mhc_testing_forward_path(int64_t B, int n, int64_t C, int *path)
{
    if (path == nullptr) return MHC_ERR_INVALID;
    MHC_TRY(check_shape(B, n, C, true));
    *path = B > 0 && takes_decode_path(B, n, C) ? 1 : 0;
    return MHC_OK;
}

int mhc_testing_check_record(int *site, int64_t *offset, int64_t *extent)
{
    if (site == nullptr || offset == nullptr || extent == nullptr) return MHC_ERR_INVALID;
    std::lock_guard<std::mutex> lock(g_check_status_mu);
    CheckRecord rec{};
    if (read_and_clear_checks(&rec) != cudaSuccess) return MHC_ERR_CUDA;
    if (g_last_check.status != 0) rec = g_last_check;  // seen first by mhc_device_status
    g_last_check = CheckRecord{};
    *site = rec.status != 0 ? rec.site : 0;
    *offset = rec.status != 0 ? rec.off : 0;
    *extent = rec.status != 0 ? rec.extent : 0;
    return MHC_OK;
}

int mhc_testing_check_selftest(void)
{
#ifdef MHC_CHECK
    float *buf = nullptr;
    if (cudaMalloc(&buf, 16 * sizeof(float)) != cudaSuccess) return MHC_ERR_CUDA;
    check_selftest_kernel<<<1, 1>>>(buf);
    cudaError_t e = cudaGetLastError();
    const cudaError_t s = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = s;
    cudaFree(buf);
    return cuda_status(e);
#else
    return MHC_ERR_UNSUPPORTED;
#endif
}

int mhc_device_status(int *status)
{
    if (status == nullptr) return MHC_ERR_INVALID;
    int st[5] = {0, 0, 0, 0, 0};
    if (read_and_clear_device_status(&st[0]) != cudaSuccess) return MHC_ERR_CUDA;
    if (read_and_clear_fused_status(&st[1]) != cudaSuccess) return MHC_ERR_CUDA;
    if (read_and_clear_decode_status(&st[2]) != cudaSuccess) return MHC_ERR_CUDA;
    if (read_and_clear_rmsnorm_gemm_status(&st[3]) != cudaSuccess) return MHC_ERR_CUDA;
    if (kCheckBuild) {
        // the records stay readable through mhc_testing_check_record
        std::lock_guard<std::mutex> lock(g_check_status_mu);
        CheckRecord rec{};
        if (read_and_clear_checks(&rec) != cudaSuccess) return MHC_ERR_CUDA;
        if (rec.status != 0 && g_last_check.status == 0) g_last_check = rec;
        st[4] = g_last_check.status;
    }
    *status = MHC_OK;
    for (int v : st)
        if (v != MHC_OK) {
            *status = v;
            break;
        }
    return MHC_OK;
}

}  // extern "C"
