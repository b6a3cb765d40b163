/*
 * mhc.h — C ABI of the GB300 (sm_103a) mHC forward library.
 *
 * Manifold-constrained hyper-connections (mHC) widen the residual stream of a
 * transformer into n parallel streams and mix them with per-token
 * coefficients.  This library computes the forward pass of that mixing as
 * analysed on the page "mHC 算法分析 & cutile 高效实现" (mHC algorithm
 * analysis and an efficient cuTile implementation), §2.1–§2.5 and §3:
 *
 *   mhc_gemm_rms        Ỹ = X·φ and r = sqrt(Σx²/(nC))          (§2.1, §2.2, §3.1)
 *   mhc_coeffs          H̃ = α·Ỹ/r + b; H_pre = σ(H̃_pre),
 *                       H_post = 2σ(H̃_post), H_res = Sinkhorn(H̃_res) (§2.3, §2.4, §3.2, §3.3)
 *   mhc_pre_apply       F_pre = Σ_i H_pre[i]·X[i]                 (§2.5)
 *   mhc_post_res_apply  X_next[i] = Σ_j H_res[i][j]·X[j] + H_post[i]·F_out (§2.5, §3.4)
 *   mhc_forward         steps 1-4b on one stream (mhc_gemm_rms_coeffs, mhc_pre_apply,
 *                       mhc_post_res_apply; for B <= 2048 steps 1-4a in one
 *                       launch, and 4b in it too for B <= 256)
 *   mhc_forward_host    mhc_forward over host buffers, copies overlapped with compute
 *   mhc_gemm_rms_coeffs steps 1-3 in one launch (mhc_gemm_rms then mhc_coeffs)
 *   mhc_rmsnorm_gemm    C = rmsnorm(A) @ B for any N (Lazy Pre-Norm, second page §2)
 *   mhc_*_f32w / _split / _f32   the fp32-weight, fp32-F_out precision variant (§5)
 *   mhc_*_e4m3          the fp8 e4m3 precision variant (§4)
 *
 * Shapes: B tokens (batch × sequence), expansion n, hidden size C,
 * K = n·C, N = n² + 2n.
 *
 * Layouts (all row-major, densely packed, no strides):
 *   X, X_next  [B][n][C] bf16   the n streams of a token side by side (= [B][K])
 *   phi_t      [N][K]    bf16   φᵀ: the projection φ ∈ R^{K×N} transposed, K contiguous
 *   F_out      [B][C]    bf16   output of the layer function F (F lies outside mHC)
 *   F_pre      [B][C]    bf16
 *   Y          [B][N]    fp32   columns [0,n) pre, [n,2n) post, [2n,N) res (row-major n×n)
 *   r          [B]       fp32
 *   bias       [N]       fp32   same column order as Y
 *   H_pre, H_post [B][n] fp32;  H_res [B][n][n] fp32, row i = output stream i
 *
 * Precision: bf16 inputs, fp32 accumulation, fp32 coefficients; bf16 outputs
 * are rounded to nearest even.
 *
 * Ownership and ordering: every pointer is a DEVICE pointer owned by the
 * caller (mhc_forward_host alone takes host activations); the library never
 * allocates, frees or keeps a pointer after a call returns.  Each call only validates its arguments and enqueues kernels on
 * `stream` (NULL = the legacy default stream); it returns without waiting.
 *
 * Argument rules (checked on the host; a failing call launches nothing):
 *   - B >= 0; B == 0 is a no-op that returns MHC_OK;
 *   - B < 2^31; 1 <= n <= 8; C >= 8, C % 8 == 0 and n*C <= 2^30;
 *     otherwise MHC_ERR_UNSUPPORTED;
 *   - pointers non-NULL (MHC_ERR_INVALID) and 16-byte aligned (MHC_ERR_ALIGN);
 *   - every device pointer (every pointer but mhc_forward_host's host
 *     activations) is device memory of the current device, as
 *     cudaPointerGetAttributes reports it: host memory, managed memory or
 *     another GPU's memory reached over peer access is MHC_ERR_INVALID;
 *   - an output may not overlap any input or another output
 *     (MHC_ERR_INVALID), except that X_next may be exactly X;
 *   - iters >= 0 (MHC_ERR_INVALID);
 *   - the current device must be compute capability 10.3 (sm_103,
 *     GB300); otherwise MHC_ERR_UNSUPPORTED.
 * Errors are returned as int status codes; no C++ exception crosses the ABI.
 * Faults inside kernels surface as CUDA errors on the caller's next
 * synchronisation; bounded waits that run out are reported by
 * mhc_device_status().
 */
#ifndef MHC_H
#define MHC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t mhc_bf16;          /* a bf16 value, stored as its 16-bit pattern */
typedef struct CUstream_st *mhc_stream_t; /* the same type as cudaStream_t */

typedef enum {
    MHC_OK = 0,
    MHC_ERR_INVALID = -1,     /* bad size, NULL pointer, overlapping buffers, iters < 0 */
    MHC_ERR_UNSUPPORTED = -2, /* n, C or device outside what the kernels handle */
    MHC_ERR_ALIGN = -3,       /* a pointer is not 16-byte aligned */
    MHC_ERR_CUDA = -4,        /* a CUDA runtime call or a kernel launch failed */
    MHC_ERR_TIMEOUT = -5,     /* a bounded device wait ran out (see mhc_device_status) */
    MHC_ERR_WORKSPACE = -6,   /* workspace NULL or smaller than mhc_workspace_bytes() */
    MHC_ERR_BOUNDS = -7       /* MHC_CHECK builds only: a device index check failed */
} mhc_status;

/* Human-readable name of a status code (static string, never NULL). */
const char *mhc_status_str(int status);

/*
 * Bytes of device workspace mhc_gemm_rms and mhc_forward need for (B, n, C)
 * on the CURRENT device (the split-K partial sums and tile counters of §5.1's
 * two-stage reduction).  Depends on the device's SM count.  Returns 0 when
 * the arguments are out of range.  The workspace needs no initialisation
 * and holds nothing between calls; calls that share one workspace must be
 * ordered (same stream, or synchronised).
 */
size_t mhc_workspace_bytes(int64_t B, int n, int64_t C);

/*
 * Step 1 — GEMM fused with the RMS reduction (§2.1, §2.2; fusion §3.1).
 *   Y[b][k] = Σ_{q<K} X[b][q]·φ[q][k]  (= Σ_q X[b][q]·phi_t[k][q]),  k < N
 *   r[b]    = sqrt( Σ_{q<K} X[b][q]² / K )   (no epsilon)
 * X is read from HBM once: the square-sum is taken from the same on-chip
 * tiles that feed the tensor cores.  Results are bitwise reproducible for a
 * given device and shape (fixed split-K summation order).  A token whose row
 * is all zero gets r = 0 (its coefficients are then not finite).
 */
int mhc_gemm_rms(const mhc_bf16 *X, const mhc_bf16 *phi_t, int64_t B, int n, int64_t C,
                 float *Y, float *r, void *workspace, size_t workspace_bytes,
                 mhc_stream_t stream);

/*
 * Steps 2–3 — coefficients (§2.3, §2.4; fusions §3.2, §3.3).
 *   H̃[b][k]   = α_seg·Y[b][k]/r[b] + bias[k]   (α_pre / α_post / α_res by column segment)
 *   H_pre     = 1/(1+e^{-H̃_pre}),  H_post = 2/(1+e^{-H̃_post})
 *   H_res     = Sinkhorn–Knopp: start from exp(H̃_res) as an n×n matrix, then
 *               `iters` times divide each row by its sum, then each column
 *               by its sum.  iters = 0 returns exp(H̃_res) unnormalised.
 * One thread per token holds the n×n block in registers through the iteration.
 */
int mhc_coeffs(const float *Y, const float *r, float alpha_pre, float alpha_post,
               float alpha_res, const float *bias, int iters, int64_t B, int n,
               float *H_pre, float *H_post, float *H_res, mhc_stream_t stream);

/*
 * Steps 1–3 in one launch: mhc_gemm_rms, then mhc_coeffs folded into the
 * GEMM's finalize.  The CTA that writes a token's Y and r forms its H_pre,
 * H_post and H_res with the same arithmetic as mhc_coeffs, so the results are
 * those of the two calls in sequence, bit for bit.  Arguments, layouts and the
 * workspace are those of mhc_gemm_rms and mhc_coeffs; mhc_forward's chain
 * runs steps 1–3 this way.
 */
int mhc_gemm_rms_coeffs(const mhc_bf16 *X, const mhc_bf16 *phi_t, float alpha_pre,
                        float alpha_post, float alpha_res, const float *bias, int iters,
                        int64_t B, int n, int64_t C, float *Y, float *r, float *H_pre,
                        float *H_post, float *H_res, void *workspace, size_t workspace_bytes,
                        mhc_stream_t stream);

/*
 * Step 4a — pre-mixing, n streams to one (§2.5 (1)):
 *   F_pre[b][c] = Σ_{i<n} H_pre[b][i]·X[b][i][c]
 */
int mhc_pre_apply(const mhc_bf16 *X, const float *H_pre, int64_t B, int n, int64_t C,
                  mhc_bf16 *F_pre, mhc_stream_t stream);

/*
 * Step 4b — residual and post mixing, fused (§2.5 (3), fusion §3.4):
 *   X_next[b][i][c] = Σ_{j<n} H_res[b][i][j]·X[b][j][c] + H_post[b][i]·F_out[b][c]
 * X is read once and X_next written once.  X_next may be exactly X (in-place
 * update); any other overlap is rejected.
 */
int mhc_post_res_apply(const mhc_bf16 *X, const mhc_bf16 *F_out, const float *H_res,
                       const float *H_post, int64_t B, int n, int64_t C, mhc_bf16 *X_next,
                       mhc_stream_t stream);

/*
 * The whole forward on `stream`, with the same argument rules and results as
 * mhc_gemm_rms, mhc_coeffs, mhc_pre_apply and mhc_post_res_apply called in
 * that order.  F_out is an input, present from the start: inside a real layer
 * it is F(F_pre), which lies outside mHC (§2.5 (2)), and such a layer calls the
 * step entry points with F between them.  X_next may be exactly X.
 *
 * Path: for B <= 2048 steps 1-4a run as one cooperative launch (the split-K
 * GEMM over every SM, a bounded grid barrier, then each CTA's fixed-order
 * reduction, coefficients and F_pre, and for B <= 256 X_next too; above 256
 * mhc_post_res_apply follows), which measured faster than the kernel chain at
 * those sizes; above 2048, the chain (mhc_gemm_rms_coeffs,
 * mhc_pre_apply, mhc_post_res_apply).  Either path is
 * deterministic; they differ in the split-K order, so Y (and what follows
 * from it) differs between them in the last bits, within the tolerances.
 */
int mhc_forward(const mhc_bf16 *X, const mhc_bf16 *phi_t, const mhc_bf16 *F_out,
                float alpha_pre, float alpha_post, float alpha_res, const float *bias,
                int iters, int64_t B, int n, int64_t C, float *Y, float *r, float *H_pre,
                float *H_post, float *H_res, mhc_bf16 *F_pre, mhc_bf16 *X_next,
                void *workspace, size_t workspace_bytes, mhc_stream_t stream);

/*
 * Bytes of DEVICE scratch mhc_forward_host needs for (B, n, C) on the current
 * device: three chunk slots of bf16 buffers for chunks of up to 1024 tokens,
 * the fp32 outputs (Y, r, H) of the whole batch and the forward workspace
 * (about 0.27 GB at B=16384, n=4, C=7168).  0 when the
 * arguments are out of range or no device is usable.
 */
size_t mhc_forward_host_scratch_bytes(int64_t B, int n, int64_t C);

/*
 * mhc_forward over HOST-resident activations:
 *   X, F_out                        host inputs   (layouts as mhc_forward)
 *   Y, r, H_pre, H_post, H_res,
 *   F_pre, X_next                   host outputs  (X_next may be exactly X)
 *   phi_t, bias                     DEVICE inputs (weights, resident)
 *   scratch                         DEVICE scratch of mhc_forward_host_scratch_bytes
 * The batch goes through the device in chunks of tokens: 256 and 512 first,
 * then chunks of 1024 (the last of them possibly shorter), then 512 and 256,
 * so that the first copy in and the last copy out, which nothing overlaps,
 * are short; a batch below 2560 tokens goes in chunks of 256 (of a quarter
 * of the batch, at least 1, below 1024 tokens), the last possibly shorter.
 * mhc_testing_host_chunks (mhc_testing.h) returns the plan.  The copy of one chunk to the device, the forward of the
 * previous one (mhc_forward's path for the chunk size) and the copy of the
 * outputs before that back to the host run concurrently on two internal copy
 * streams and `stream`.  Every copy is one cudaMemcpyAsync.  Results equal
 * mhc_forward's on the same chunks bit for bit (tokens are independent, §2.3).
 *
 * Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister) for
 * the copies to overlap; pageable memory is accepted and copies synchronously.
 * The call is stream-ordered: it starts after the work already on `stream`,
 * and work enqueued on `stream` afterwards starts only once every output is in
 * host memory (synchronise `stream` before reading them).  Calls on one device
 * are serialised on the library's copy streams; do not touch the host buffers
 * or the scratch until then.
 *
 * Rules of mhc_forward, plus: the activation pointers must be host memory and
 * phi_t, bias and scratch device memory (MHC_ERR_INVALID otherwise);
 * scratch_bytes < mhc_forward_host_scratch_bytes gives MHC_ERR_WORKSPACE.
 */
int mhc_forward_host(const mhc_bf16 *X, const mhc_bf16 *phi_t, const mhc_bf16 *F_out,
                     float alpha_pre, float alpha_post, float alpha_res, const float *bias,
                     int iters, int64_t B, int n, int64_t C, float *Y, float *r, float *H_pre,
                     float *H_post, float *H_res, mhc_bf16 *F_pre, mhc_bf16 *X_next,
                     void *scratch, size_t scratch_bytes, mhc_stream_t stream);

/*
 * fp32-weight precision variant.  The page's optimised benchmark (§5) keeps
 * the weight in fp32 (run as TF32 by its MMA) and F_out in fp32 while X stays
 * bf16.  Here the fp32 φᵀ is split once into bf16 pairs and the bf16 tensor
 * cores run twice as many columns:
 *   mhc_split_phi       phi_t [N][K] fp32 -> phi_split [2N][K] bf16: row 2k is
 *                       the bf16 value nearest φᵀ[k], row 2k+1 the bf16 value
 *                       nearest the remainder; hi + lo is within about 2^-17
 *                       relative of the fp32 weight (TF32 keeps 2^-11);
 *   mhc_gemm_rms_split  mhc_gemm_rms with phi_split: Ỹ[k] = acc[2k] + acc[2k+1]
 *                       (same workspace as mhc_gemm_rms);
 *   mhc_post_res_apply_f32  mhc_post_res_apply with F_out [B][C] fp32;
 *   mhc_forward_f32w    the forward with both (X, F_pre, X_next bf16): like
 *                       mhc_forward, steps 1-4a (1-4b up to 256) in one launch
 *                       for B <= 2048, else the kernel chain; workspace of
 *                       mhc_workspace_bytes.
 * Rules, layouts and status codes otherwise as the bf16 calls.
 */
int mhc_split_phi(const float *phi_t, int n, int64_t C, mhc_bf16 *phi_split, mhc_stream_t stream);
int mhc_gemm_rms_split(const mhc_bf16 *X, const mhc_bf16 *phi_split, int64_t B, int n, int64_t C,
                       float *Y, float *r, void *workspace, size_t workspace_bytes,
                       mhc_stream_t stream);
int mhc_post_res_apply_f32(const mhc_bf16 *X, const float *F_out, const float *H_res,
                           const float *H_post, int64_t B, int n, int64_t C, mhc_bf16 *X_next,
                           mhc_stream_t stream);
int mhc_forward_f32w(const mhc_bf16 *X, const mhc_bf16 *phi_split, const float *F_out,
                     float alpha_pre, float alpha_post, float alpha_res, const float *bias,
                     int iters, int64_t B, int n, int64_t C, float *Y, float *r, float *H_pre,
                     float *H_post, float *H_res, mhc_bf16 *F_pre, mhc_bf16 *X_next,
                     void *workspace, size_t workspace_bytes, mhc_stream_t stream);

/*
 * fp8 e4m3 precision variant (the precision of the page's first benchmark,
 * §4): X [B][K], φᵀ [N][K], F_out, F_pre [B][C] and X_next [B][K] are e4m3
 * codes (OCP E4M3: bias 7, 3 mantissa bits, largest finite 448, no
 * infinities), one byte each; Y, r, b and H stay fp32.  The GEMM runs
 * tcgen05 kind::f8f6f4 (e4m3 × e4m3, fp32 accumulate) on 128-value K stages;
 * the square sum decodes the same tiles; the apply kernels decode exactly,
 * mix in f16 (2^-11 rounding, well below e4m3's 2^-4; partial sums beyond
 * ±65504, possible only for an unnormalised H_res, saturate) and round the
 * outputs to nearest even, saturating to ±448.
 * Rules of the bf16 calls, plus C % 16 == 0 (MHC_ERR_UNSUPPORTED otherwise);
 * the workspace is mhc_workspace_bytes(B, n, C).  mhc_forward_e4m3 always runs
 * the kernel chain (GEMM with the coefficients, then the two applies).
 */
int mhc_gemm_rms_e4m3(const uint8_t *X, const uint8_t *phi_t, int64_t B, int n, int64_t C,
                      float *Y, float *r, void *workspace, size_t workspace_bytes,
                      mhc_stream_t stream);
int mhc_pre_apply_e4m3(const uint8_t *X, const float *H_pre, int64_t B, int n, int64_t C,
                       uint8_t *F_pre, mhc_stream_t stream);
int mhc_post_res_apply_e4m3(const uint8_t *X, const uint8_t *F_out, const float *H_res,
                            const float *H_post, int64_t B, int n, int64_t C, uint8_t *X_next,
                            mhc_stream_t stream);
int mhc_forward_e4m3(const uint8_t *X, const uint8_t *phi_t, const uint8_t *F_out,
                     float alpha_pre, float alpha_post, float alpha_res, const float *bias,
                     int iters, int64_t B, int n, int64_t C, float *Y, float *r, float *H_pre,
                     float *H_post, float *H_res, uint8_t *F_pre, uint8_t *X_next,
                     void *workspace, size_t workspace_bytes, mhc_stream_t stream);

/*
 * C = rmsnorm(A) @ B, the "Lazy Pre-Norm" fusion of page "Towards Free
 * Normalization: Fusing Normalization into GEMM and Attention Kernels"
 * (PyTorch blog), §2:
 *   rstd[m] = 1 / sqrt(Σ_q A[m][q]² / K + eps),  C[m][n] = (Σ_q A[m][q]·B[q][n])·rstd[m]
 * which equals (A·rstd) @ B; the square sums are reduced from the tiles the
 * tensor cores read, so A is read from HBM once, and rstd is applied to the
 * accumulator.  mhc_gemm_rms is the skinny, eps-free case of the same
 * computation (there the scaling is left to mhc_coeffs).
 *
 * Layouts (row-major, densely packed):
 *   A    [M][K] bf16
 *   B_t  [N][K] bf16   Bᵀ, K contiguous (a linear layer's weight [out][in])
 *   C    [M][N] bf16   fp32 accumulation and scaling, rounded to nearest even
 * Rules: M >= 0 (M == 0 is a no-op); M < 2^31, 8 <= K <= 2^30 and
 * 8 <= N <= 2^24, K and N multiples of 8 (MHC_ERR_UNSUPPORTED); eps finite and >= 0 (MHC_ERR_INVALID);
 * pointers non-NULL and 16-byte aligned; C may not overlap A or B_t.
 * workspace: mhc_rmsnorm_gemm_workspace_bytes(M, K, N) bytes of device memory
 * (0 when every CTA gets whole output tiles; then workspace may be NULL).
 * Results are deterministic (a fixed summation order).
 */
size_t mhc_rmsnorm_gemm_workspace_bytes(int64_t M, int64_t K, int64_t N);
int mhc_rmsnorm_gemm(const mhc_bf16 *A, const mhc_bf16 *B_t, int64_t M, int64_t K, int64_t N,
                     float eps, mhc_bf16 *C, void *workspace, size_t workspace_bytes,
                     mhc_stream_t stream);

/*
 * Size of the built-in scratch array of mhc_gemm_rms_noalloc: 16 MiB, held in
 * device memory by every GPU that loads this library, until the process
 * exits.  A (B, n, C) fits when the GEMM's own split-K scratch (the part of
 * mhc_workspace_bytes that mhc_gemm_rms checks) is at most this; on a 152-SM
 * GB300 that scratch does not depend on C: n=4 fits up to B = 148,224 tokens,
 * n=8 up to B = 32,256.  mhc_workspace_bytes itself may be larger: it also
 * covers the other forward paths.
 */
#define MHC_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/*
 * mhc_gemm_rms without a workspace argument: the same computation, kernel and
 * results, with the split-K scratch taken from the library's own fixed device
 * array instead of caller memory.  The mHC page has no counterpart to this
 * call; it exists for callers that cannot allocate device memory where they
 * call it — code running inside a host framework that owns all device memory
 * through its own pool, or a latency-critical path where a cudaMalloc (which
 * can synchronise the device) is not acceptable.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *
 * - Same argument rules and status codes as mhc_gemm_rms.  A problem that
 *   needs more than MHC_NOALLOC_SCRATCH_BYTES of scratch is rejected with
 *   MHC_ERR_WORKSPACE before anything is launched.
 * - Every call looks up the array's device address in the current context
 *   (the lookup allocates nothing), so a context created anew is served too.
 *   The first call on a device loads the library's device code there: make it
 *   before any stream capture on that device.
 * - Every call on a device shares the one array and it keeps the last call's
 *   contents (each call clears what must start at zero itself).  Calls that
 *   overlap on the GPU — on different streams, or from different threads
 *   without ordering — race on it: order them.
 */
int mhc_gemm_rms_noalloc(const mhc_bf16 *X, const mhc_bf16 *phi_t, int64_t B, int n, int64_t C,
                         float *Y, float *r, mhc_stream_t stream);

/*
 * Reads and clears the device status word of the current device: MHC_OK, or
 * MHC_ERR_TIMEOUT when a bounded wait inside a kernel ran out since the last
 * read (the kernel then stopped early, so its outputs are not valid).  A
 * library built with -DMHC_CHECK also reports MHC_ERR_BOUNDS when a device
 * index check failed since the last read (the access was skipped, so the
 * outputs are not valid either); the default build has no such checks.
 * Blocks until all prior work on the device has finished.  Returns MHC_OK or
 * MHC_ERR_CUDA; the status is written to *status.
 */
int mhc_device_status(int *status);

#ifdef __cplusplus
}
#endif

#endif /* MHC_H */
