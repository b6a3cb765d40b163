"""The fp8 e4m3 precision variant (page "mHC 算法分析 & cutile 高效实现", §4
benchmark precision) through the C ABI against the fp64 oracle on the same
e4m3 inputs.

Tolerance of an e4m3 output (3 mantissa bits): half an ulp, 2^-4·|ref|, plus
half the subnormal step 2^-10, plus the f16 mixing ((n+2) roundings of 2^-11,
taken as 2^-7 of Σ|terms|); past ±448 the output saturates.  Y: 1e-5·Σ|x·φ| + 1e-6 as for bf16 (e4m3 products are exact in
fp32).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import H_TOL, R_REL, assert_abs, assert_rel, cuda_ok, for_all_rows, host64
from synth import WORKLOADS

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]

mhc = pytest.importorskip("gemm_rms_sinkhorn_gb300")


def dev8(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).cuda()


def host8(t):
    return t.cpu().numpy().view(np.uint8)


def dec(codes):
    return synth.e4m3_bits_to_f32(codes).astype(np.float64)


def assert_e4m3_close(got_codes, ref, what, absdot=None):
    got = dec(got_codes)
    ref = np.asarray(ref, dtype=np.float64).reshape(got.shape)
    sat = np.abs(ref) >= 464.0
    assert np.all(got[sat] == np.sign(ref[sat]) * 448.0), what + ": saturation"
    bound = 2.0 ** -4 * np.abs(ref) + 2.0 ** -10 + 1e-6
    if absdot is not None:
        bound = bound + 2.0 ** -7 * absdot.reshape(got.shape)
    err = np.abs(got - ref)
    ok = sat | (err <= bound)
    assert np.all(ok), "%s: max err/bound %.3g" % (what, float(np.max(np.where(sat, 0, err / bound))))


def mix_absdots(X, Fo, ref, n, C):
    """Σ|terms| of F_pre and of X_next, from the oracle's coefficients."""
    B = X.shape[0]
    x = np.abs(dec(X)).reshape(B, n, C)
    f = np.abs(dec(Fo)).reshape(B, C)
    fp = np.einsum("bi,bic->bc", np.abs(ref["H_pre"]), x)
    xn = np.einsum("bij,bjc->bic", np.abs(ref["H_res"]), x) + np.abs(ref["H_post"])[:, :, None] * f[:, None, :]
    return fp, xn.reshape(B, n * C)


def inputs(B, n, C, seed, phi_std=0.02):
    N, K = n * n + 2 * n, n * C
    X = synth.normal_e4m3((B, K), seed, 0, 1.0)
    Fo = synth.normal_e4m3((B, C), seed, 1, 1.0)
    phi_t = synth.normal_e4m3((N, K), seed, 2, phi_std)
    bias = synth.normal_f32((N,), seed, 3, 0.1)
    return X, phi_t, Fo, bias


def gemm(X, phi_t, n, C):
    B, N = X.shape[0], phi_t.shape[0]
    Y = torch.empty(B, N, device="cuda")
    r = torch.empty(B, device="cuda")
    mhc.mhc_gemm_rms_e4m3(dev8(X), dev8(phi_t), B, n, C, Y, r, mhc.workspace(B, n, C))
    torch.cuda.synchronize()
    return host64(Y), host64(r)


@pytest.mark.parametrize("B,n,C", [(1, 1, 16), (5, 4, 16), (130, 8, 32), (300, 4, 7168)])
def test_gemm_e4m3_exact_integers(B, n, C):
    """Integers in [-8, 8] are exact in e4m3 and every partial sum is exact in fp32."""
    N, K = n * n + 2 * n, n * C
    X = synth.f32_to_e4m3_bits(synth.bf16_bits_to_f32(synth.int_bf16((B, K), 81, 0, -8, 8)))
    P = synth.f32_to_e4m3_bits(synth.bf16_bits_to_f32(synth.int_bf16((N, K), 81, 2, -8, 8)))
    Y, r = gemm(X, P, n, C)
    Yr = dec(X) @ dec(P).T
    assert np.array_equal(Y, Yr)
    assert_rel(r, np.sqrt((dec(X) ** 2).mean(axis=1)), 2.0 ** -22, "r")


def test_pre_apply_e4m3_one_hot_reproduces_every_code():
    """H_pre = e_i: F_pre = X[i] re-encoded, bit for bit, for all finite codes."""
    n, C = 2, 256
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[~np.isnan(synth.e4m3_bits_to_f32(codes))]
    row = np.resize(codes, C)
    X = np.stack([np.concatenate([row, np.roll(row, 7)])] * 3)  # B = 3 tokens
    for i in range(n):
        Hp = np.zeros((3, n), np.float32)
        Hp[:, i] = 1.0
        F = torch.empty(3, C, dtype=torch.uint8, device="cuda")
        mhc.mhc_pre_apply_e4m3(dev8(X), torch.from_numpy(Hp).cuda(), 3, n, C, F)
        torch.cuda.synchronize()
        want = X.reshape(3, n, C)[:, i, :]
        got = host8(F)
        zero = dec(want) == 0  # -0 and +0 both encode a zero product
        assert np.array_equal(got[~zero], want[~zero]) and np.all(dec(got[zero]) == 0)


# every n from 1 to 8 (each is its own instantiation of the three e4m3 kernels),
# ragged token tiles, C a multiple of 16 but not of 64
@pytest.mark.parametrize("B,n,C", [(64, 4, 256), (7, 1, 16), (300, 8, 512), (129, 3, 4096),
                                   (200, 2, 256), (65, 5, 272), (129, 6, 48), (257, 7, 16)])
def test_forward_e4m3_matches_oracle(B, n, C):
    X, P, Fo, bias = inputs(B, n, C, seed=82)
    out = mhc.alloc_outputs(B, n, C)
    F_pre = torch.empty(B, C, dtype=torch.uint8, device="cuda")
    X_next = torch.empty(B, n * C, dtype=torch.uint8, device="cuda")
    mhc.mhc_forward_e4m3(dev8(X), dev8(P), dev8(Fo), 0.01, 0.01, 0.01,
                         torch.from_numpy(bias).cuda(), 20, B, n, C, out["Y"], out["r"],
                         out["H_pre"], out["H_post"], out["H_res"], F_pre, X_next, out["ws"])
    torch.cuda.synchronize()
    ref = oracle.forward_e4m3(X, np.ascontiguousarray(P.T), Fo, n, C, 0.01, 0.01, 0.01, bias, 20)
    Yb = 1e-5 * (np.abs(dec(X)) @ np.abs(dec(P)).T) + 1e-6
    assert np.all(np.abs(host64(out["Y"]) - ref["Y"]) <= Yb), "Y"
    assert_rel(host64(out["r"]), ref["r"], R_REL, "r")
    for k in ("H_pre", "H_post", "H_res"):
        assert_abs(host64(out[k]), ref[k], H_TOL, k)
    fp, xn = mix_absdots(X, Fo, ref, n, C)
    assert_e4m3_close(host8(F_pre), ref["F_pre"], "F_pre", fp)
    assert_e4m3_close(host8(X_next), ref["X_next"], "X_next", xn)


def test_forward_e4m3_prefill_every_token():
    """B=16384, n=4, C=7168 in e4m3 (470 MB of X): every token against the oracle, a
    token range per host core."""
    wl = WORKLOADS["prefill"]
    B, n, C = wl.B, wl.n, wl.C
    X, P, Fo, bias = inputs(B, n, C, seed=83)
    out = mhc.alloc_outputs(B, n, C)
    F_pre = torch.empty(B, C, dtype=torch.uint8, device="cuda")
    X_next = torch.empty(B, n * C, dtype=torch.uint8, device="cuda")
    mhc.mhc_forward_e4m3(dev8(X), dev8(P), dev8(Fo), wl.alpha_pre, wl.alpha_post, wl.alpha_res,
                         torch.from_numpy(bias).cuda(), wl.iters, B, n, C, out["Y"], out["r"],
                         out["H_pre"], out["H_post"], out["H_res"], F_pre, X_next, out["ws"])
    torch.cuda.synchronize()
    g = {k: host64(out[k]) for k in ("Y", "r", "H_pre", "H_post", "H_res")}
    g_fp, g_xn = host8(F_pre), host8(X_next)
    PT = np.ascontiguousarray(P.T)
    absP = np.abs(dec(P)).T

    def part(lo, hi):
        ref = oracle.forward_e4m3(X[lo:hi], PT, Fo[lo:hi], n, C, wl.alpha_pre, wl.alpha_post,
                                  wl.alpha_res, bias, wl.iters)
        what = " (tokens %d-%d)" % (lo, hi - 1)
        Yb = 1e-5 * (np.abs(dec(X[lo:hi])) @ absP) + 1e-6
        assert np.all(np.abs(g["Y"][lo:hi] - ref["Y"]) <= Yb), "Y" + what
        assert_rel(g["r"][lo:hi], ref["r"], R_REL, "r" + what)
        for k in ("H_pre", "H_post", "H_res"):
            assert_abs(g[k][lo:hi], ref[k], H_TOL, k + what)
        fp, xn = mix_absdots(X[lo:hi], Fo[lo:hi], ref, n, C)
        assert_e4m3_close(g_fp[lo:hi], ref["F_pre"], "F_pre" + what, fp)
        assert_e4m3_close(g_xn[lo:hi], ref["X_next"], "X_next" + what, xn)

    for_all_rows(B, part)
