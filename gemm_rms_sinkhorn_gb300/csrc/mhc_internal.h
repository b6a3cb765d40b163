// Launchers shared between the translation units of the library.  Arguments
// have already been validated by the C ABI layer (api.cu) when these run.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace mhc {

// Launches `kernel` with programmatic stream serialisation: its CTAs may
// start while the previous kernel in the stream finishes, and every kernel
// of this library calls pdl_wait() before it touches global memory, so the
// launch latency and prologue overlap the predecessor without changing the
// stream order of memory accesses.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// As launch_pdl, and cooperative: every CTA of the grid is resident at once
// (the launch fails otherwise), so CTAs may wait on one another.
template <typename... KArgs, typename... Args>
cudaError_t launch_coop_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// N = n² + 2n coefficient columns per token.
inline int num_coeffs(int n) { return n * n + 2 * n; }

// Cached per-device facts (SM count, compute capability).
struct DeviceInfo {
    int device = -1;
    int num_sms = 0;
    int cc_major = 0;
    int cc_minor = 0;
};
cudaError_t current_device_info(DeviceInfo *info);

// ---- step 1: GEMM + RMS (gemm_rms.cu)
// Every wait inside the GEMM kernel gives up after this much GPU time.
constexpr uint64_t kWaitLimitNs = 4000000000ull;
size_t gemm_rms_workspace_bytes(int64_t B, int n, int64_t C, int num_sms);
// Steps 2 and 3 folded into the GEMM's finalize: with H_pre non-null, the CTA
// that writes a token's Y and r also forms its H_pre, H_post and H_res
// (token_coeffs, the coefficient kernel's computation, so the same bits).
struct CoefArgs {
    const float *bias = nullptr;
    float a_pre = 0.f, a_post = 0.f, a_res = 0.f;
    int iters = 0, n = 0;
    float *H_pre = nullptr, *H_post = nullptr, *H_res = nullptr;
};
// stall_stage >= 0 is a test hook: CTA 0 leaves that pipeline stage unfilled.
cudaError_t launch_gemm_rms(const uint16_t *X, const uint16_t *phi_t, int64_t B, int n,
                            int64_t C, float *Y, float *r, void *workspace, int num_sms,
                            cudaStream_t stream, uint64_t wait_limit_ns = kWaitLimitNs,
                            int64_t stall_stage = -1, const CoefArgs &coef = CoefArgs{});
cudaError_t read_and_clear_device_status(int *status);
// The fp32-weight form: phi_split [2N][K] bf16 (hi and remainder of each
// fp32 weight column, interleaved) from launch_split_phi; the same Y and r.
cudaError_t launch_gemm_rms_split(const uint16_t *X, const uint16_t *phi_split, int64_t B, int n,
                                  int64_t C, float *Y, float *r, void *workspace, int num_sms,
                                  cudaStream_t stream, const CoefArgs &coef = CoefArgs{});
cudaError_t launch_split_phi(const float *phi_t, int n, int64_t C, uint16_t *phi_split,
                             cudaStream_t stream);
// The fp8 form: X [B][K] and phi_t [N][K] as e4m3 codes (kind::f8f6f4 MMAs,
// 128 K values per stage); the same Y, r and workspace.
cudaError_t launch_gemm_rms_e4m3(const uint8_t *X, const uint8_t *phi_t, int64_t B, int n,
                                 int64_t C, float *Y, float *r, void *workspace, int num_sms,
                                 cudaStream_t stream, const CoefArgs &coef = CoefArgs{});

// Tensor map of a 2-D bf16 tensor [rows][cols] (cols contiguous): boxes of
// box_rows × 64 elements, 128-byte swizzle, zero fill out of bounds.
bool make_tmap(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_rows);

// ---- steps 1-4a in one persistent kernel, X read once (fused_pre.cu)
bool fused_pre_eligible(int64_t B, int n, int64_t C, int num_sms);
size_t fused_pre_workspace_bytes(int64_t B, int n, int64_t C, int num_sms);
cudaError_t launch_fused_pre(const uint16_t *X, const uint16_t *phi_t, float a_pre, float a_post,
                             float a_res, const float *bias, int iters, int64_t B, int n,
                             int64_t C, float *Y, float *r, float *H_pre, float *H_post,
                             float *H_res, uint16_t *F_pre, void *workspace, int num_sms,
                             cudaStream_t stream);
cudaError_t read_and_clear_fused_status(int *status);

// ---- steps 1-4a in one cooperative launch for small batches (decode_pre.cu)
bool decode_pre_eligible(int64_t B, int n, int64_t C);
size_t decode_pre_workspace_bytes(int64_t B, int n, int64_t C, int num_sms);
// barrier_extra > 0 is a test hook: the grid barrier waits for that many
// arrivals more than there are CTAs, so every CTA's wait runs out.  split:
// phi_t is the fp32-weight form (bf16 pairs, 2N rows).
// Steps 1-4a in one cooperative launch (small batches), and step 4b too when
// X_next is not NULL.  F_out is bf16, or fp32 when split (the fp32-weight
// forward); X_next may be X.
cudaError_t launch_decode_pre(const uint16_t *X, const uint16_t *phi_t, float a_pre, float a_post,
                              float a_res, const float *bias, int iters, int64_t B, int n,
                              int64_t C, float *Y, float *r, float *H_pre, float *H_post,
                              float *H_res, uint16_t *F_pre, const void *F_out, uint16_t *X_next,
                              void *workspace, int num_sms, cudaStream_t stream,
                              uint64_t wait_limit_ns = kWaitLimitNs, int barrier_extra = 0,
                              bool split = false);
cudaError_t read_and_clear_decode_status(int *status);

// ---- the whole forward on device buffers (api.cu), arguments already valid
// Workspace of every forward path (and of mhc_gemm_rms), whichever is largest.
size_t forward_workspace_bytes(int64_t B, int n, int64_t C, int num_sms);
// mhc_forward's own choice of path: the one-launch steps 1-4a kernel for small
// batches, else the kernel chain; then the X_next kernel.
cudaError_t run_forward_device(const uint16_t *X, const uint16_t *phi_t, const uint16_t *F_out,
                               float a_pre, float a_post, float a_res, const float *bias,
                               int iters, int64_t B, int n, int64_t C, float *Y, float *r,
                               float *H_pre, float *H_post, float *H_res, uint16_t *F_pre,
                               uint16_t *X_next, void *workspace, int num_sms,
                               cudaStream_t stream);

// ---- the forward over host buffers (host_pipeline.cu)
// Tokens a chunk carries through the device: small enough that the first
// copy in and the last copy out, which nothing overlaps, stay short, large
// enough that each copy runs at link speed.
constexpr int64_t kHostChunkTokens = 1024;
constexpr int kHostSlots = 3;               // chunks in flight (copy in, compute, copy out)
// Byte sizes (each 256-byte aligned) of one chunk slot's bf16 buffers (x,
// f_out, f_pre), of the batch-wide fp32 outputs (y, r, h_*), of the forward
// workspace shared by the chunks, and of the whole scratch.
struct HostChunkLayout {
    int64_t chunk_tokens;
    size_t x, f_out, f_pre, y, r, h_pre, h_post, h_res, slot, workspace, total;
};
HostChunkLayout host_chunk_layout(int64_t B, int n, int64_t C, int num_sms);
cudaError_t run_forward_host(const uint16_t *X, const uint16_t *phi_t, const uint16_t *F_out,
                             float a_pre, float a_post, float a_res, const float *bias, int iters,
                             int64_t B, int n, int64_t C, float *Y, float *r, float *H_pre,
                             float *H_post, float *H_res, uint16_t *F_pre, uint16_t *X_next,
                             void *scratch, int num_sms, cudaStream_t stream);

// ---- step 4 on e4m3 activations (apply_e4m3.cu); C % 16 == 0
cudaError_t launch_pre_apply_e4m3(const uint8_t *X, const float *H_pre, int64_t B, int n,
                                  int64_t C, uint8_t *F_pre, cudaStream_t stream);
cudaError_t launch_post_res_apply_e4m3(const uint8_t *X, const uint8_t *F_out, const float *H_res,
                                       const float *H_post, int64_t B, int n, int64_t C,
                                       uint8_t *X_next, cudaStream_t stream);

// ---- C = rmsnorm(A) @ B, Lazy Pre-Norm (rmsnorm_gemm.cu)
size_t rmsnorm_gemm_workspace_bytes(int64_t M, int64_t K, int64_t N, int num_sms);
cudaError_t launch_rmsnorm_gemm(const uint16_t *A, const uint16_t *B_t, int64_t M, int64_t K,
                                int64_t N, float eps, uint16_t *C, void *workspace, int num_sms,
                                cudaStream_t stream);
cudaError_t read_and_clear_rmsnorm_gemm_status(int *status);

// ---- steps 2-3: coefficients + Sinkhorn (coeffs.cu)
cudaError_t launch_coeffs(const float *Y, const float *r, float a_pre, float a_post, float a_res,
                          const float *bias, int iters, int64_t B, int n, float *H_pre,
                          float *H_post, float *H_res, cudaStream_t stream);
// Test hook: out[i] = the reciprocal the Sinkhorn normalisations and sigmoids use, of in[i].
cudaError_t launch_recip(const float *in, float *out, int64_t count, cudaStream_t stream);

// ---- step 4: apply kernels (apply.cu)
cudaError_t launch_pre_apply(const uint16_t *X, const float *H_pre, int64_t B, int n, int64_t C,
                             uint16_t *F_pre, cudaStream_t stream);
cudaError_t launch_post_res_apply(const uint16_t *X, const uint16_t *F_out, const float *H_res,
                                  const float *H_post, int64_t B, int n, int64_t C,
                                  uint16_t *X_next, cudaStream_t stream);
// The same with F_out in fp32.
cudaError_t launch_post_res_apply_f32(const uint16_t *X, const float *F_out, const float *H_res,
                                      const float *H_post, int64_t B, int n, int64_t C,
                                      uint16_t *X_next, cudaStream_t stream);

}  // namespace mhc
