/*
 * mhc_testing.h — test hooks of the GB300 mHC forward library.  Not part of
 * the stable API; used by the library's own tests to exercise paths that
 * normal inputs never reach.
 */
#ifndef MHC_TESTING_H
#define MHC_TESTING_H

#include "mhc.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * mhc_gemm_rms with two changes, so that the bounded waits inside the kernel
 * can be seen to work without faulting or hanging the GPU:
 *   - CTA 0 leaves pipeline stage number `stall_stage` (counted from 0 over
 *     that CTA's whole run) unfilled, so its consumers wait on it in vain;
 *   - every wait in the kernel gives up after `wait_limit_ns` nanoseconds of
 *     GPU time (clamped to [1 ms, 4 s]) instead of 4 s.
 * When a wait runs out the kernel records MHC_ERR_TIMEOUT in the device status
 * word (read with mhc_device_status), lets its issued copies land, drains
 * its tensor-core work, frees its tensor memory and returns; the CUDA context
 * stays usable.  Y and r are then not valid.  Argument rules and return codes
 * are those of mhc_gemm_rms; stall_stage < 0 stalls nothing.
 */
int mhc_testing_gemm_rms_stalled(const mhc_bf16 *X, const mhc_bf16 *phi_t, int64_t B, int n,
                                 int64_t C, float *Y, float *r, void *workspace,
                                 size_t workspace_bytes, int64_t stall_stage,
                                 uint64_t wait_limit_ns, mhc_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MHC_TESTING_H */
