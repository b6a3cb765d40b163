"""The fp32-weight precision variant (page "mHC 算法分析 & cutile 高效实现",
§5: X bf16, weight fp32 (TF32 there), other inputs fp32) through the C ABI
against the fp64 oracle's float-input functions.

Tolerances: Y within 1e-5·Σ|x·φ| + 1e-6 (fp32 accumulation of exact products,
plus the hi/lo split of φ, which is within about 2^-17 of φ); the others as in
the bf16 tests (gpu_util).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import (H_TOL, R_REL, assert_abs, assert_bf16_close, assert_rel, cuda_ok,
                      dev_bf16, dev_f32, f64, for_all_rows, host64, host_bits, host_outputs)
from synth import WORKLOADS, make_inputs

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]

mhc = pytest.importorskip("gemm_rms_sinkhorn_gb300")

SHAPES = [(1, 1, 8), (3, 2, 8), (5, 4, 16), (65, 5, 264), (129, 6, 40), (257, 7, 8),
          (200, 4, 264), (130, 8, 72), (3, 3, 24), (1, 4, 7168), (128, 4, 7168), (300, 8, 512)]


def phi_f32(n, C, seed):
    """fp32 φᵀ [N, K] ~ N(0, 0.02²), not rounded to bf16."""
    N, K = n * n + 2 * n, n * C
    return synth.normal_f32((N, K), seed, 2, 0.02)


def split(phi_t):
    N, K = phi_t.shape
    n = next(m for m in range(1, 9) if m * m + 2 * m == N)
    out = torch.empty(2 * N, K, dtype=torch.bfloat16, device="cuda")
    mhc.mhc_split_phi(dev_f32(phi_t), n, K // n, out)
    torch.cuda.synchronize()
    return out


def assert_Y_f32(got, ref, X_bits, phi_t):
    bound = 1e-5 * (np.abs(f64(X_bits)) @ np.abs(phi_t.astype(np.float64)).T) + 1e-6
    err = np.abs(got - ref)
    assert np.all(err <= bound), "Y: max err/bound %.3g" % float(np.max(err / bound))


def test_split_phi_is_nearest_hi_and_remainder():
    phi = phi_f32(4, 512, 71)
    s = host_bits(split(phi)).reshape(phi.shape[0], 2, -1)
    hi_want = synth.f32_to_bf16_bits(phi)
    assert np.array_equal(s[:, 0], hi_want)
    hi = synth.bf16_bits_to_f32(hi_want).astype(np.float32)
    lo_want = synth.f32_to_bf16_bits((phi - hi).astype(np.float32))
    assert np.array_equal(s[:, 1], lo_want)
    recon = hi.astype(np.float64) + synth.bf16_bits_to_f32(lo_want).astype(np.float64)
    assert np.all(np.abs(recon - phi) <= 2.0 ** -16 * np.abs(phi) + 1e-30)


@pytest.mark.parametrize("B,n,C", SHAPES)
def test_gemm_rms_split_matches_oracle(B, n, C):
    X = synth.normal_bf16((B, n * C), 72, 0)
    phi = phi_f32(n, C, 72)
    N = phi.shape[0]
    Y = torch.empty(B, N, device="cuda")
    r = torch.empty(B, device="cuda")
    mhc.mhc_gemm_rms_split(dev_bf16(X), split(phi), B, n, C, Y, r, mhc.workspace(B, n, C))
    torch.cuda.synchronize()
    Yr, rr = oracle.gemm_rms_f64phi(X, np.ascontiguousarray(phi.T).astype(np.float64), n, C)
    assert_Y_f32(host64(Y), Yr, X, phi)
    assert_rel(host64(r), rr, R_REL, "r")


@pytest.mark.parametrize("inplace", [False, True])
def test_post_res_apply_f32_matches_oracle(inplace):
    B, n, C = 65, 4, 264
    X = synth.normal_bf16((B, n * C), 73, 0)
    Fo = synth.normal_f32((B, C), 73, 1, 1.0)
    Hr = oracle.sinkhorn(synth.normal_f32((B, n, n), 73, 9, 1.0), 20).astype(np.float32)
    Hq = 2.0 * (np.abs(synth.normal_f32((B, n), 73, 8, 0.5)) % 1.0)
    Xd = dev_bf16(X)
    out = Xd if inplace else torch.empty_like(Xd)
    mhc.mhc_post_res_apply_f32(Xd, dev_f32(Fo), dev_f32(Hr), dev_f32(Hq), B, n, C, out)
    torch.cuda.synchronize()
    ref = oracle.post_res_apply_f64F(X, Fo.astype(np.float64), Hr.astype(np.float64),
                                     Hq.astype(np.float64), n, C)
    assert_bf16_close(host64(out), ref, "X_next")


def forward_f32w(wl, seed):
    """The fp32-weight forward on every token, against the oracle a token range per host core."""
    inp = make_inputs(wl, seed=seed, parts=("X", "bias"))
    X = inp["X"]
    phi = phi_f32(wl.n, wl.C, seed)
    Fo = synth.normal_f32((wl.B, wl.C), seed, 1, 1.0)
    out = mhc.alloc_outputs(wl.B, wl.n, wl.C)
    mhc.mhc_forward_f32w(dev_bf16(X), split(phi), dev_f32(Fo), wl.alpha_pre, wl.alpha_post,
                         wl.alpha_res, dev_f32(inp["bias"]), wl.iters, wl.B, wl.n, wl.C, out["Y"],
                         out["r"], out["H_pre"], out["H_post"], out["H_res"], out["F_pre"],
                         out["X_next"], out["ws"])
    torch.cuda.synchronize()
    g = host_outputs(out)
    phi_kn = np.ascontiguousarray(phi.T).astype(np.float64)

    def part(lo, hi):
        ref = oracle.forward_f64w(X[lo:hi], phi_kn, Fo[lo:hi].astype(np.float64), wl.n, wl.C,
                                  wl.alpha_pre, wl.alpha_post, wl.alpha_res, inp["bias"],
                                  wl.iters)
        what = " (tokens %d-%d)" % (lo, hi - 1)
        assert_Y_f32(g["Y"][lo:hi], ref["Y"], X[lo:hi], phi)
        assert_rel(g["r"][lo:hi], ref["r"], R_REL, "r" + what)
        for k in ("H_pre", "H_post", "H_res"):
            assert_abs(g[k][lo:hi], ref[k], H_TOL, k + what)
        assert_bf16_close(f64(g["F_pre"][lo:hi]), ref["F_pre"], "F_pre" + what)
        assert_bf16_close(f64(g["X_next"][lo:hi]), ref["X_next"], "X_next" + what)

    for_all_rows(wl.B, part)


@pytest.mark.parametrize("name", ["tiny", "decode1", "decode128"])
def test_forward_f32w_matches_oracle(name):
    forward_f32w(WORKLOADS[name], seed=74)


def test_forward_f32w_7b_every_token():
    forward_f32w(WORKLOADS["7b"], seed=75)


def test_forward_f32w_wider_n8():
    forward_f32w(WORKLOADS["wider"].with_(B=300), seed=76)


@pytest.mark.parametrize("n", [1, 2, 3, 5, 6, 7, 8])
def test_forward_f32w_chain_every_n(n):
    """Above 2048 tokens the forward takes the kernel chain, whose split-weight GEMM forms
    the coefficients in its finalize: one GEMM width per n (2N padded to 16)."""
    wl = WORKLOADS["tiny"].with_(B=3200, n=n, C=64, bias_std=0.3)
    forward_f32w(wl, seed=77 + n)


@pytest.mark.parametrize("n", [1, 2, 3, 5, 6, 7])
def test_forward_f32w_decode_every_n(n):
    """Up to 2048 tokens the forward takes the one-launch small-batch path with the
    split weight (its partial rows hold both halves of each column pair): every n."""
    wl = WORKLOADS["tiny"].with_(B=100, n=n, C=72, bias_std=0.3)
    forward_f32w(wl, seed=90 + n)
