// Device index checks of the MHC_CHECK build.
//
// Built with -DMHC_CHECK, each kernel asks in_range(site, off, len, extent)
// before a global access it addresses by computed offsets: whether elements
// [off, off + len) lie inside a buffer of `extent` elements (an empty range
// always passes).  A failed check records the first failure of its
// translation unit (site, offset, extent) and returns false, and the caller
// skips the access; the kernel runs on.  No trap, no fault: the host reads
// the record through mhc_device_status (MHC_ERR_BOUNDS) and
// mhc_testing_check_record.  In the default build every check is the
// constant true and compiles away.
//
// Sites are numbered per source file: 100s apply.cu, 200s apply_e4m3.cu, 300s
// coeffs.cu, 400s gemm_rms.cu, 500s fused_pre.cu, 600s decode_pre.cu, 700s
// rmsnorm_gemm.cu, 900 the check build's self-test.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace mhc {

constexpr int kStatusBounds = -7;  // MHC_ERR_BOUNDS

struct CheckRecord {
    int status;  // 0, or kStatusBounds after a failed check
    int site;    // the first failing site
    long long off;
    long long extent;
};

using CheckReader = cudaError_t (*)(CheckRecord *);

// Host side (api.cu): every translation unit with checks registers the
// reader of its record when the library loads.
bool register_check_reader(CheckReader reader);

#ifdef MHC_CHECK
constexpr bool kCheckBuild = true;

namespace {

__device__ CheckRecord g_check;  // one per translation unit

__device__ __noinline__ void record_bounds(int site, long long off, long long extent)
{
    if (atomicCAS(&g_check.status, 0, kStatusBounds) == 0) {
        g_check.site = site;
        g_check.off = off;
        g_check.extent = extent;
    }
}

cudaError_t read_and_clear_check(CheckRecord *out)
{
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    if ((e = cudaMemcpyFromSymbol(out, g_check, sizeof *out)) != cudaSuccess) return e;
    const CheckRecord zero{};
    return cudaMemcpyToSymbol(g_check, &zero, sizeof zero);
}

[[maybe_unused]] const bool g_check_registered = register_check_reader(&read_and_clear_check);

}  // namespace

__device__ __forceinline__ bool in_range(int site, int64_t off, int64_t len, int64_t extent)
{
    if (len == 0) return true;  // an empty range touches nothing, wherever it starts
    if (off >= 0 && len > 0 && off + len <= extent) return true;
    record_bounds(site, off, extent);
    return false;
}
#else
constexpr bool kCheckBuild = false;

__device__ __forceinline__ constexpr bool in_range(int, int64_t, int64_t, int64_t) { return true; }
#endif

}  // namespace mhc
