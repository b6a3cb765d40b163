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

/*
 * mhc_forward with steps 1-4a in one persistent kernel that reads X from HBM
 * once for both the projection GEMM and the pre-mixing: chunks of token tiles
 * small enough to stay in L2, several CTAs per tile with a deterministic
 * fixed-order reduction of their partial sums, and the pre-apply re-reading
 * each tile's X with bulk copies.  Same arguments, rules, outputs and
 * tolerances as mhc_forward (the split-K partition differs, so Y differs in
 * rounding).  Returns MHC_ERR_UNSUPPORTED for shapes the kernel does not take
 * (fewer than two 128-token tiles, or K too short to split over the CTAs of
 * a tile).  Measured on GB300 it is not yet faster than mhc_forward: the
 * second read of X mostly misses L2, so mhc_forward does not use it.
 */
int mhc_testing_forward_fused(const mhc_bf16 *X, const mhc_bf16 *phi_t, const mhc_bf16 *F_out,
                              float alpha_pre, float alpha_post, float alpha_res,
                              const float *bias, int iters, int64_t B, int n, int64_t C, float *Y,
                              float *r, float *H_pre, float *H_post, float *H_res,
                              mhc_bf16 *F_pre, mhc_bf16 *X_next, void *workspace,
                              size_t workspace_bytes, mhc_stream_t stream);

/*
 * mhc_forward forced onto the kernel chain (mhc_gemm_rms_coeffs,
 * mhc_pre_apply, mhc_post_res_apply), which mhc_forward itself takes only
 * above its small-batch threshold.  Same arguments, rules and outputs as
 * mhc_forward.
 */
int mhc_testing_forward_chain(const mhc_bf16 *X, const mhc_bf16 *phi_t, const mhc_bf16 *F_out,
                              float alpha_pre, float alpha_post, float alpha_res,
                              const float *bias, int iters, int64_t B, int n, int64_t C, float *Y,
                              float *r, float *H_pre, float *H_post, float *H_res,
                              mhc_bf16 *F_pre, mhc_bf16 *X_next, void *workspace,
                              size_t workspace_bytes, mhc_stream_t stream);

/*
 * mhc_forward forced onto the small-batch path: steps 1-4a in one cooperative
 * launch (the split-K GEMM over all SMs, a bounded grid barrier, then each
 * CTA's fixed-order reduction, coefficients and F_pre of its share of the
 * channels), with X_next in it for B <= 256 and the X_next kernel after it
 * above.  mhc_forward takes this path by itself for B <= 2048; this hook
 * takes it for any B <= 4096.  Same arguments, rules and outputs as
 * mhc_forward; MHC_ERR_UNSUPPORTED for B > 4096.
 */
int mhc_testing_forward_decode(const mhc_bf16 *X, const mhc_bf16 *phi_t, const mhc_bf16 *F_out,
                               float alpha_pre, float alpha_post, float alpha_res,
                               const float *bias, int iters, int64_t B, int n, int64_t C,
                               float *Y, float *r, float *H_pre, float *H_post, float *H_res,
                               mhc_bf16 *F_pre, mhc_bf16 *X_next, void *workspace,
                               size_t workspace_bytes, mhc_stream_t stream);

/*
 * mhc_testing_forward_decode whose grid barrier waits for one arrival more
 * than there are CTAs, so every CTA's wait runs out after `wait_limit_ns`
 * nanoseconds of GPU time (clamped to [1 ms, 4 s]).  Each CTA then records
 * MHC_ERR_TIMEOUT in the device status word (read with mhc_device_status)
 * and returns without writing Y, r, H or F_pre, nor X_next up to 256 tokens;
 * above that the X_next kernel still runs on whatever H_res and H_post hold.
 * The barrier's words are left clear, so the next call on the same workspace
 * works normally.  The CUDA context stays usable.
 */
int mhc_testing_forward_decode_stalled(const mhc_bf16 *X, const mhc_bf16 *phi_t,
                                       const mhc_bf16 *F_out, float alpha_pre, float alpha_post,
                                       float alpha_res, const float *bias, int iters, int64_t B,
                                       int n, int64_t C, float *Y, float *r, float *H_pre,
                                       float *H_post, float *H_res, mhc_bf16 *F_pre,
                                       mhc_bf16 *X_next, void *workspace, size_t workspace_bytes,
                                       mhc_stream_t stream, uint64_t wait_limit_ns);

/*
 * out[i] = the reciprocal the Sinkhorn–Knopp normalisations and the sigmoids
 * multiply by, of in[i]: the hardware's approximate reciprocal (rcp.approx,
 * subnormal inputs and results flushed to zero).  `count` fp32 values, device
 * pointers, 16-byte aligned, not overlapping.  MHC_ERR_INVALID for count < 0
 * or a NULL pointer.
 */
int mhc_testing_recip(const float *in, float *out, int64_t count, mhc_stream_t stream);

/*
 * The chunk plan of mhc_forward_host for a batch of B tokens (host only, no
 * device needed): *count = the number of chunks, and the first
 * min(*count, capacity) token counts, in order, go to sizes[] (host memory).
 * MHC_ERR_INVALID for B < 0, capacity < 0, a NULL count, or a NULL sizes
 * with capacity > 0.
 */
int mhc_testing_host_chunks(int64_t B, int64_t *sizes, int64_t capacity, int64_t *count);

/*
 * Turns the device-memory pointer checks of the device entry points off
 * (on = 0) or on (on != 0), process-wide, and returns the previous setting.
 * They are on unless this is called; switching them off only serves to time
 * what they cost on the host.  The other argument checks always run.
 */
int mhc_testing_memory_checks(int on);

/*
 * 1 if the library was built with -DMHC_CHECK (device index checks that
 * record a failure and skip the access instead of faulting), else 0.
 */
int mhc_testing_check_build(void);

/*
 * Reads and clears the device index-check records of every translation unit
 * (waits for the device first).  *site = the first failing site (0: none),
 * *offset and *extent = its element offset and the buffer's element count.
 * MHC_ERR_INVALID for a NULL pointer, MHC_ERR_CUDA if a copy fails.  In the
 * default build every record is empty.
 */
int mhc_testing_check_record(int *site, int64_t *offset, int64_t *extent);

/*
 * Check build only: launches one thread that asks for element `extent` of a
 * 16-element device buffer it owns (one past the end), which the check
 * refuses and records as site 900 without touching memory.  Returns MHC_OK
 * after the launch, MHC_ERR_UNSUPPORTED in the default build (which would
 * not check), MHC_ERR_CUDA on a launch failure.
 */
int mhc_testing_check_selftest(void);

/*
 * Host only (no device needed): the path mhc_forward and mhc_forward_f32w take
 * for (B, n, C), written to *path: 1 = the one-launch kernel (small batches,
 * B <= 2048: steps 1-4a, and 4b with them up to 256 tokens), 0 = the kernel
 * chain (GEMM with the coefficients, pre apply, X_next).  B = 0 gives 0.
 * Status codes as mhc_forward's shape checks; MHC_ERR_INVALID for a NULL path.
 */
int mhc_testing_forward_path(int64_t B, int n, int64_t C, int *path);

#ifdef __cplusplus
}
#endif

#endif /* MHC_TESTING_H */
