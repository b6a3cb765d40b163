// mhc_gemm_rms_noalloc: mhc_gemm_rms for callers that cannot allocate device
// memory.  The split-K scratch of the GEMM + RMS kernel (tile tickets and
// partial sums) lives in one file-scope device array of fixed size instead of
// a caller-provided workspace.  The array is part of the library's device
// image, so every GPU that loads the library holds it until the process
// exits.  All calls share it: calls that overlap on the GPU (for example on
// two streams at once) race on it and must be ordered by the caller.
#include <cuda_runtime.h>

#include <cstdint>

#include "mhc.h"

namespace {

constexpr size_t kScratchBytes = MHC_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of g_noalloc_scratch in the current context.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// with the caller's device current, on every call: the lookup allocates
// nothing, and a context created anew (after cudaDeviceReset, say) may hold
// the array at another address, so no address is kept between calls.  The
// first lookup on a device loads the library's device code there, which is why
// the first call on a device should come before any stream capture.  Returns
// nullptr when the lookup fails.
void *current_device_scratch()
{
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
        cudaGetLastError();  // not sticky; clear it
        return nullptr;
    }
    return p;
}

}  // namespace

extern "C" int mhc_gemm_rms_noalloc(const mhc_bf16 *X, const mhc_bf16 *phi_t, int64_t B, int n,
                                    int64_t C, float *Y, float *r, mhc_stream_t stream)
{
    if (B == 0)  // no device work: only the shape rules apply
        return mhc_gemm_rms(X, phi_t, 0, n, C, Y, r, nullptr, 0, stream);
    void *scratch = current_device_scratch();
    if (scratch == nullptr) return MHC_ERR_CUDA;
    // Same validation and kernel as mhc_gemm_rms; a problem whose scratch
    // need exceeds kScratchBytes is rejected there with MHC_ERR_WORKSPACE
    // before anything is launched.  The kernel launch clears the tile
    // tickets that must start at zero; the partial sums are written before
    // they are read.
    return mhc_gemm_rms(X, phi_t, B, n, C, Y, r, scratch, kScratchBytes, stream);
}
