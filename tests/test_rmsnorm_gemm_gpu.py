"""C = rmsnorm(A) @ B (page "Towards Free Normalization: Fusing Normalization
into GEMM and Attention Kernels", §2, Lazy Pre-Norm) through the C ABI against
the fp64 oracle, which normalises first and then multiplies.

Tolerance per element: the bf16 rounding of C (half an ulp, 2^-9 relative,
taken as 2^-8) plus fp32 accumulation over K of exact bf16 products
(1e-5 of Σ_q |A·B|·rstd), as for the mHC GEMM.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import cuda_ok, dev_bf16, f64, host64, sample_rows

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]

mhc = pytest.importorskip("gemm_rms_sinkhorn_gb300")


def inputs(M, K, N, seed, b_std=0.05):
    A = synth.normal_bf16((M, K), seed, 0)
    B_t = synth.normal_bf16((N, K), seed, 2, b_std)
    return A, B_t


def run(A, B_t, eps):
    M, K = A.shape
    C = mhc.rmsnorm_gemm(dev_bf16(A), dev_bf16(B_t), eps)
    torch.cuda.synchronize()
    return C


def check(C_gpu, A, B_t, eps, rows=None):
    sel = np.arange(A.shape[0]) if rows is None else np.asarray(rows)
    ref = oracle.rmsnorm_gemm(A[sel], np.ascontiguousarray(B_t.T), eps)
    got = host64(C_gpu)[sel]
    Af, Bf = f64(A[sel]), f64(B_t)
    rstd = 1.0 / np.sqrt((Af ** 2).mean(axis=1) + eps)
    absdot = (np.abs(Af) @ np.abs(Bf).T) * rstd[:, None]
    bound = 2.0 ** -8 * np.abs(ref) + 1e-5 * absdot + 1e-30
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got))
    assert np.all(err <= bound), "max err/bound %.3g" % float(np.max(err / bound))


# whole-tile (>= 152 tiles) and split-K (fewer tiles than SMs) schedules, every
# column-tile width (32, 64, 128, 256), ragged rows, columns and K blocks
# (shapes 9-11: an odd number of row tiles, a column tile cut inside its second
# half).  With 256-column tiles and X = ceil(M/256)·ceil(N/256), X >= 152 with
# K >= 4096 takes the 256-row tiles (ragged rows, K blocks and columns; then a
# last group of 4 row tiles after two of 8 in the grouped tile order; then 4 row
# tiles in all, one short group)
SHAPES = [(128, 64, 32), (300, 72, 40), (1000, 520, 200), (4096, 512, 1024),
          (8192, 256, 8), (2048, 1024, 256), (513, 4104, 96), (20000, 128, 64),
          (2000, 520, 2560), (19000, 200, 696), (2500, 1000, 4000), (4000, 4104, 2504),
          (5000, 4096, 2048), (1000, 4096, 10240)]


@pytest.mark.parametrize("M,K,N", SHAPES)
def test_rmsnorm_gemm_matches_oracle(M, K, N):
    A, B_t = inputs(M, K, N, seed=41)
    C = run(A, B_t, 1e-5)
    rows = None if M * K * N <= 3e9 else sample_rows(M, 96)
    check(C, A, B_t, 1e-5, rows)
    again = run(A, B_t, 1e-5)
    assert torch.equal(C, again)  # fixed summation order: bitwise reproducible


@pytest.mark.parametrize("eps", [0.0, 1e-5, 1.0])
def test_rmsnorm_gemm_eps_and_zero_rows(eps):
    M, K, N = 260, 192, 96
    A, B_t = inputs(M, K, N, seed=42)
    if eps > 0:
        A[7] = 0  # rstd = 1/sqrt(eps) is finite: the row of C is zero
    C = run(A, B_t, eps)
    check(C, A, B_t, eps)
    if eps > 0:
        assert not bool(C[7].any())


def test_rmsnorm_gemm_large_whole_tiles_sampled():
    """16384 × 2048 → 2048 (1024 whole tiles of 128 × 256), rows sampled."""
    M, K, N = 16384, 2048, 2048
    A, B_t = inputs(M, K, N, seed=43, b_std=0.02)
    C = run(A, B_t, 1e-5)
    check(C, A, B_t, 1e-5, sample_rows(M, 48))


def test_rmsnorm_gemm_row_scale_invariance():
    """eps = 0: rmsnorm(2A) = rmsnorm(A), and 2A is exact in bf16, so C is identical."""
    M, K, N = 200, 256, 64
    A, B_t = inputs(M, K, N, seed=44)
    A2 = synth.f32_to_bf16_bits(2.0 * synth.bf16_bits_to_f32(A))
    assert torch.equal(run(A, B_t, 0.0), run(A2, B_t, 0.0))


def test_rmsnorm_gemm_status_clean():
    assert mhc.mhc_device_status() == mhc.MHC_OK
