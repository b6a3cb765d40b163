"""GPU parity: every kernel of the library, through the C ABI, against the
fp64 oracle on the same seeded inputs (page "mHC 算法分析 & cutile 高效实现",
§2.1–§2.5).  Tolerances are in ``gpu_util``.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import (H_TOL, R_REL, assert_abs, assert_bf16_close, assert_rel, assert_Y_close,
                      cuda_ok, dev_bf16, dev_f32, f64, for_all_rows, host64, host_bits,
                      host_outputs, phi_KN)
from synth import WORKLOADS, make_inputs

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]

mhc = pytest.importorskip("gemm_rms_sinkhorn_gb300")

# (B, n, C): ragged tiles (B % 128 != 0), ragged K blocks (n*C % 64 != 0), every N padding
ODD_SHAPES = [(1, 1, 8), (3, 2, 8), (5, 4, 16), (65, 5, 264), (129, 6, 40), (257, 7, 8),
              (200, 4, 264), (130, 8, 72), (3, 3, 24)]


def gemm_gpu(X_bits, phi_t_bits, n, C):
    B = X_bits.shape[0]
    N = n * n + 2 * n
    Y = torch.empty(B, N, dtype=torch.float32, device="cuda")
    r = torch.empty(B, dtype=torch.float32, device="cuda")
    ws = mhc.workspace(B, n, C)
    mhc.mhc_gemm_rms(dev_bf16(X_bits), dev_bf16(phi_t_bits), B, n, C, Y, r, ws)
    torch.cuda.synchronize()
    return host64(Y), host64(r)


# ------------------------------------------------------------- step 1


@pytest.mark.parametrize("B,n,C", ODD_SHAPES + [(1, 4, 7168), (128, 4, 7168), (300, 8, 512)])
def test_gemm_rms_exact_integers(B, n, C):
    """Integer X, φ in [-2, 2]: Ỹ and Σx² are exact in fp32, so Y must match bit for bit."""
    K, N = n * C, n * n + 2 * n
    X = synth.int_bf16((B, K), 101, 0, -2, 2)
    phi_t = synth.int_bf16((N, K), 101, 2, -2, 2)
    Y, r = gemm_gpu(X, phi_t, n, C)
    Yr, rr = oracle.gemm_rms(X, phi_KN(phi_t), n, C)
    assert np.array_equal(Y, Yr), "max |dY| %g" % np.max(np.abs(Y - Yr))
    assert_rel(r, rr, 2.0 ** -22, "r (1 ulp)")


@pytest.mark.parametrize("name", ["tiny", "decode1", "decode8", "decode32", "decode128", "7b"])
def test_gemm_rms_workloads(name):
    wl = WORKLOADS[name]
    inp = make_inputs(wl, seed=0, parts=("X", "phi_t"))
    Y, r = gemm_gpu(inp["X"], inp["phi_t"], wl.n, wl.C)
    Yr, rr = oracle.gemm_rms(inp["X"], phi_KN(inp["phi_t"]), wl.n, wl.C)
    assert_Y_close(Y, Yr, inp["X"], inp["phi_t"])
    assert_rel(r, rr, R_REL, "r")


@pytest.mark.parametrize("B,n,C", ODD_SHAPES)
def test_gemm_rms_odd_shapes(B, n, C):
    K, N = n * C, n * n + 2 * n
    X = synth.normal_bf16((B, K), 7, 0)
    phi_t = synth.normal_bf16((N, K), 7, 2, 0.02)
    Y, r = gemm_gpu(X, phi_t, n, C)
    Yr, rr = oracle.gemm_rms(X, phi_KN(phi_t), n, C)
    assert_Y_close(Y, Yr, X, phi_t)
    assert_rel(r, rr, R_REL, "r")


def test_gemm_rms_deterministic():
    wl = WORKLOADS["decode32"]
    inp = make_inputs(wl, seed=1, parts=("X", "phi_t"))
    a = gemm_gpu(inp["X"], inp["phi_t"], wl.n, wl.C)
    b = gemm_gpu(inp["X"], inp["phi_t"], wl.n, wl.C)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ---------------------------------------------------------- steps 2-3


def coeffs_gpu(Y, r, al, bias, iters, n):
    B = Y.shape[0]
    Hp = torch.empty(B, n, device="cuda")
    Hq = torch.empty(B, n, device="cuda")
    Hr = torch.empty(B, n, n, device="cuda")
    mhc.mhc_coeffs(dev_f32(Y), dev_f32(r), al[0], al[1], al[2], dev_f32(bias), iters, B, n,
                   Hp, Hq, Hr)
    torch.cuda.synchronize()
    return host64(Hp), host64(Hq), host64(Hr)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("iters", [0, 1, 5, 20, 50])
def test_coeffs(n, iters):
    B, N = 300, n * n + 2 * n
    Y = synth.normal_f32((B, N), 200 + n, 9, 3.0)
    r = np.abs(synth.normal_f32(B, 300 + n, 9, 1.0)) + 0.05
    bias = synth.normal_f32(N, 400 + n, 3, 0.5)
    al = (0.7, -0.3, 0.9)
    Hp, Hq, Hr = coeffs_gpu(Y, r, al, bias, iters, n)
    # the oracle gets the very same fp32 values, widened
    Op, Oq, Or = oracle.coeffs(Y.astype(np.float64), r.astype(np.float64), np.float32(al[0]),
                               np.float32(al[1]), np.float32(al[2]), bias.astype(np.float64),
                               iters)
    assert_abs(Hp, Op, H_TOL, "H_pre")
    assert_abs(Hq, Oq, H_TOL, "H_post")
    # |H̃| reaches ~100 here, where σ rounds to exactly 0 or 1: closed ranges
    assert (Hp >= 0).all() and (Hp <= 1).all() and (Hq >= 0).all() and (Hq <= 2).all()
    if iters == 0:
        # raw exp(H̃_res): relative agreement inside fp32's normal range; beyond
        # it (|H̃| > ~88) fp32 underflows to zero/denormals or overflows to inf
        # fp32 rounding of H̃ itself (a few ulps of |H̃|) becomes a relative
        # error of exp: allow 1e-6 + 8·2^-24·(1 + |H̃|)
        normal = (Or >= 1e-30) & (Or <= 3e38)
        tol = 1e-6 + 8 * 2.0 ** -24 * (1 + np.abs(np.log(Or[normal])))
        rel = np.abs(Hr[normal] - Or[normal]) / Or[normal]
        assert (rel <= tol).all(), "exp(H̃_res): worst rel/tol %.3f" % np.max(rel / tol)
        assert (Hr[Or < 1e-30] <= 1e-29).all()
        assert np.isposinf(Hr[Or > 3.5e38]).all()
    else:
        assert_abs(Hr, Or, H_TOL, "H_res")
        assert_abs(Hr.sum(axis=1), np.ones((B, n)), 1e-5, "H_res column sums")


def test_coeffs_closed_forms():
    """α = 0: H_pre = σ(b), H_post = 2σ(b), and a constant res bias gives H_res = 1/n."""
    n, B = 4, 70
    N = n * n + 2 * n
    bias = np.zeros(N, dtype=np.float32)
    bias[:n] = np.log(3.0)
    bias[n:2 * n] = -np.log(3.0)
    bias[2 * n:] = 0.25
    Y = synth.normal_f32((B, N), 5, 9, 1.0)
    r = np.ones(B, dtype=np.float32)
    Hp, Hq, Hr = coeffs_gpu(Y, r, (0.0, 0.0, 0.0), bias, 20, n)
    assert_abs(Hp, np.full((B, n), 0.75), 1e-6, "σ(ln 3)")
    assert_abs(Hq, np.full((B, n), 0.5), 1e-6, "2σ(-ln 3)")
    assert_abs(Hr, np.full((B, n, n), 0.25), 1e-6, "1/n")


# ------------------------------------------------------------- step 4


@pytest.mark.parametrize("B,n,C", ODD_SHAPES + [(64, 4, 7168)])
def test_pre_apply(B, n, C):
    X = synth.normal_bf16((B, n * C), 11, 0)
    Hp = np.abs(synth.normal_f32((B, n), 12, 9, 0.5)) % 1.0
    F = torch.empty(B, C, dtype=torch.bfloat16, device="cuda")
    mhc.mhc_pre_apply(dev_bf16(X), dev_f32(Hp), B, n, C, F)
    torch.cuda.synchronize()
    assert_bf16_close(host64(F), oracle.pre_apply(X, Hp.astype(np.float64), n, C), "F_pre")


def test_pre_apply_onehot_is_exact():
    B, n, C = 9, 4, 136
    X = synth.normal_bf16((B, n * C), 13, 0)
    for i in range(n):
        Hp = np.zeros((B, n), dtype=np.float32)
        Hp[:, i] = 1.0
        F = torch.empty(B, C, dtype=torch.bfloat16, device="cuda")
        mhc.mhc_pre_apply(dev_bf16(X), dev_f32(Hp), B, n, C, F)
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(F), X.reshape(B, n, C)[:, i, :])


def post_gpu(X, Fo, Hr, Hq, n, C, inplace=False):
    B = Fo.shape[0]
    Xd = dev_bf16(X)
    out = Xd if inplace else torch.empty_like(Xd)
    mhc.mhc_post_res_apply(Xd, dev_bf16(Fo), dev_f32(Hr), dev_f32(Hq), B, n, C, out)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("B,n,C", ODD_SHAPES + [(64, 4, 7168)])
@pytest.mark.parametrize("inplace", [False, True])
def test_post_res_apply(B, n, C, inplace):
    X = synth.normal_bf16((B, n * C), 21, 0)
    Fo = synth.normal_bf16((B, C), 21, 1)
    Hr = oracle.sinkhorn(synth.normal_f32((B, n, n), 22, 9, 1.0), 20).astype(np.float32)
    Hq = 2.0 * (np.abs(synth.normal_f32((B, n), 23, 9, 0.5)) % 1.0)
    out = post_gpu(X, Fo, Hr, Hq, n, C, inplace)
    ref = oracle.post_res_apply(X, Fo, Hr.astype(np.float64), Hq.astype(np.float64), n, C)
    assert_bf16_close(host64(out), ref, "X_next")


# Wide n (5..8) runs one wave of resident blocks that walk the tokens: these
# batches exceed a wave's token rows (at most 152 SMs x 4 blocks at these
# widths), so every block mixes several tokens through its double buffer.
WIDE_WALK_SHAPES = [(3000, 5, 264), (2500, 6, 40), (1900, 7, 8), (4100, 8, 72), (700, 8, 4096)]


@pytest.mark.parametrize("B,n,C", WIDE_WALK_SHAPES)
def test_pre_apply_wide_walk(B, n, C):
    X = synth.normal_bf16((B, n * C), 14, 0)
    Hp = np.abs(synth.normal_f32((B, n), 15, 9, 0.5)) % 1.0
    F = torch.empty(B, C, dtype=torch.bfloat16, device="cuda")
    mhc.mhc_pre_apply(dev_bf16(X), dev_f32(Hp), B, n, C, F)
    torch.cuda.synchronize()
    assert_bf16_close(host64(F), oracle.pre_apply(X, Hp.astype(np.float64), n, C), "F_pre")


@pytest.mark.parametrize("B,n,C", WIDE_WALK_SHAPES)
@pytest.mark.parametrize("inplace", [False, True])
def test_post_res_apply_wide_walk(B, n, C, inplace):
    X = synth.normal_bf16((B, n * C), 25, 0)
    Fo = synth.normal_bf16((B, C), 25, 1)
    Hr = oracle.sinkhorn(synth.normal_f32((B, n, n), 26, 9, 1.0), 20).astype(np.float32)
    Hq = 2.0 * (np.abs(synth.normal_f32((B, n), 27, 9, 0.5)) % 1.0)
    out = post_gpu(X, Fo, Hr, Hq, n, C, inplace)
    ref = oracle.post_res_apply(X, Fo, Hr.astype(np.float64), Hq.astype(np.float64), n, C)
    assert_bf16_close(host64(out), ref, "X_next")


def test_wide_apply_token_walk_is_exact():
    """Every token its own one-hot H_pre and permutation H_res: a coefficient
    taken from the wrong token or the wrong half of the double buffer moves
    whole streams, which an exact comparison sees."""
    B, n, C = 3001, 8, 64
    X = synth.normal_bf16((B, n * C), 28, 0)
    Fo = synth.normal_bf16((B, C), 28, 1)
    rng = np.random.default_rng(29)
    sel = rng.integers(0, n, size=B)
    Hp = np.zeros((B, n), dtype=np.float32)
    Hp[np.arange(B), sel] = 1.0
    F = torch.empty(B, C, dtype=torch.bfloat16, device="cuda")
    mhc.mhc_pre_apply(dev_bf16(X), dev_f32(Hp), B, n, C, F)
    torch.cuda.synchronize()
    Xr = X.reshape(B, n, C)
    assert np.array_equal(host_bits(F), Xr[np.arange(B), sel, :])
    perms = np.stack([rng.permutation(n) for _ in range(B)])
    Hr = np.zeros((B, n, n), dtype=np.float32)
    for i in range(n):
        Hr[np.arange(B), i, perms[:, i]] = 1.0
    out = post_gpu(X, Fo, Hr, np.zeros((B, n), dtype=np.float32), n, C)
    want = np.take_along_axis(Xr, perms[:, :, None], axis=1)
    assert np.array_equal(host_bits(out).reshape(B, n, C), want)


@pytest.mark.parametrize("n", [5, 8])
def test_pre_apply_long_walk_is_exact(n):
    """The wide pre kernel runs 32 waves of blocks, one token per block up to
    that many rows; 160001 tokens of 64 channels (8-channel items, 128-thread
    blocks, at most 16 resident per SM) make every block row walk about two
    tokens, so the register-held next H_pre is used.  One-hot H_pre per token:
    a coefficient from the wrong token moves a whole stream."""
    B, C = 160001, 64
    X = synth.normal_bf16((B, n * C), 30, 0)
    sel = np.random.default_rng(31).integers(0, n, size=B)
    Hp = np.zeros((B, n), dtype=np.float32)
    Hp[np.arange(B), sel] = 1.0
    F = torch.empty(B, C, dtype=torch.bfloat16, device="cuda")
    mhc.mhc_pre_apply(dev_bf16(X), dev_f32(Hp), B, n, C, F)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(F), X.reshape(B, n, C)[np.arange(B), sel, :])


def test_post_res_apply_permutation_is_exact():
    B, n, C = 5, 3, 64
    X = synth.normal_bf16((B, n * C), 24, 0)
    Fo = synth.normal_bf16((B, C), 24, 1)
    pi = [2, 0, 1]
    Hr = np.zeros((B, n, n), dtype=np.float32)
    for i in range(n):
        Hr[:, i, pi[i]] = 1.0
    out = post_gpu(X, Fo, Hr, np.zeros((B, n), dtype=np.float32), n, C)
    assert np.array_equal(host_bits(out).reshape(B, n, C), X.reshape(B, n, C)[:, pi, :])


# ------------------------------------------------------------ forward


FORWARD_PATHS = {"fused": "mhc_testing_forward_fused", "chain": "mhc_testing_forward_chain",
                 "decode": "mhc_testing_forward_decode"}


def forward_gpu(inp, wl, inplace=False, path="auto"):
    """mhc_forward ("auto": the library picks the path) or one forced path."""
    X = dev_bf16(inp["X"])
    B = X.shape[0]
    out = mhc.alloc_outputs(B, wl.n, wl.C)
    if inplace:
        out["X_next"] = X
    args = (X, dev_bf16(inp["phi_t"]), dev_bf16(inp["F_out"]), wl.alpha_pre, wl.alpha_post,
            wl.alpha_res, dev_f32(inp["bias"]), wl.iters)
    if path == "auto":
        mhc.forward(*args, wl.n, wl.C, out=out)
    else:
        getattr(mhc, FORWARD_PATHS[path])(*args, B, wl.n, wl.C, out["Y"], out["r"],
                                          out["H_pre"], out["H_post"], out["H_res"],
                                          out["F_pre"], out["X_next"], out["ws"])
    torch.cuda.synchronize()
    return out


def check_forward(out, inp, wl, rows=None):
    sel = slice(None) if rows is None else torch.as_tensor(rows, device="cuda")
    X = inp["X"] if rows is None else inp["X"][rows]
    Fo = inp["F_out"] if rows is None else inp["F_out"][rows]
    ref = oracle.forward(X, phi_KN(inp["phi_t"]), Fo, wl.n, wl.C, wl.alpha_pre, wl.alpha_post,
                         wl.alpha_res, inp["bias"], wl.iters)
    g = {k: host64(out[k][sel]) for k in ("Y", "r", "H_pre", "H_post", "H_res", "F_pre",
                                           "X_next")}
    assert_Y_close(g["Y"], ref["Y"], X, inp["phi_t"])
    assert_rel(g["r"], ref["r"], R_REL, "r")
    assert_abs(g["H_pre"], ref["H_pre"], H_TOL, "H_pre")
    assert_abs(g["H_post"], ref["H_post"], H_TOL, "H_post")
    assert_abs(g["H_res"], ref["H_res"], H_TOL, "H_res")
    assert_bf16_close(g["F_pre"], ref["F_pre"], "F_pre")
    assert_bf16_close(g["X_next"], ref["X_next"], "X_next")


def check_properties(out, wl):
    """Facts that hold at any size: ranges, Sinkhorn column sums, finite outputs."""
    Hp, Hq, Hr = out["H_pre"], out["H_post"], out["H_res"]
    assert bool(((Hp > 0) & (Hp < 1)).all()) and bool(((Hq > 0) & (Hq < 2)).all())
    if wl.iters > 0:
        colsum = Hr.double().sum(dim=1)
        assert float((colsum - 1).abs().max()) <= 1e-5
    assert bool(torch.isfinite(out["r"]).all()) and bool((out["r"] > 0).all())
    for k in ("F_pre", "X_next"):
        assert bool(torch.isfinite(out[k].float()).all())


@pytest.mark.parametrize("name", ["tiny", "decode1", "decode8", "decode32", "decode128", "7b"])
def test_forward_full_oracle(name):
    wl = WORKLOADS[name]
    inp = make_inputs(wl, seed=0)
    out = forward_gpu(inp, wl)
    check_forward_all_rows(out, inp, wl)
    check_properties(out, wl)


def check_forward_all_rows(out, inp, wl):
    """Every token of a large workload against the oracle, a token range per host core."""
    g = host_outputs(out)
    phi = phi_KN(inp["phi_t"])

    def part(lo, hi):
        ref = oracle.forward(inp["X"][lo:hi], phi, inp["F_out"][lo:hi], wl.n, wl.C,
                             wl.alpha_pre, wl.alpha_post, wl.alpha_res, inp["bias"], wl.iters)
        what = " (tokens %d-%d)" % (lo, hi - 1)
        assert_Y_close(g["Y"][lo:hi], ref["Y"], inp["X"][lo:hi], inp["phi_t"], "Y" + what)
        assert_rel(g["r"][lo:hi], ref["r"], R_REL, "r" + what)
        for k in ("H_pre", "H_post", "H_res"):
            assert_abs(g[k][lo:hi], ref[k], H_TOL, k + what)
        assert_bf16_close(f64(g["F_pre"][lo:hi]), ref["F_pre"], "F_pre" + what)
        assert_bf16_close(f64(g["X_next"][lo:hi]), ref["X_next"], "X_next" + what)

    for_all_rows(wl.B, part)


@pytest.mark.parametrize("name", ["wider_it5", "wider", "wider_it50"])
def test_forward_wider_every_token(name):
    """B=8192, n=8, C=4096, Student-t X: every token and every element."""
    wl = WORKLOADS[name]
    inp = make_inputs(wl, seed=0)
    out = forward_gpu(inp, wl)
    check_forward_all_rows(out, inp, wl)
    check_properties(out, wl)


def test_forward_prefill_every_token():
    """B=16384, n=4, C=7168 in the launch configuration the benchmark times: every token
    and every element against the oracle."""
    wl = WORKLOADS["prefill"]
    inp = make_inputs(wl, seed=0)
    out = forward_gpu(inp, wl)
    check_forward_all_rows(out, inp, wl)
    check_properties(out, wl)
    # run again: bitwise identical (fixed split-K order)
    Y0, X0 = out["Y"].clone(), out["X_next"].clone()
    out2 = forward_gpu(inp, wl)
    assert torch.equal(Y0, out2["Y"]) and torch.equal(X0, out2["X_next"])


# steps 1-3 in one launch (the GEMM's finalize forms the coefficients): tiles
# split over many CTAs, whole tiles owned by one CTA (K = 64: one unit each),
# every n, ragged last tiles
GEMM_COEFF_SHAPES = [(64, 4, 256), (1000, 4, 7168), (300, 8, 512), (5, 3, 24), (777, 1, 1000),
                     (2048, 6, 2048), (40000, 1, 64), (20000, 2, 32), (700, 5, 168), (900, 7, 96)]


@pytest.mark.parametrize("B,n,C,iters", [s + (20,) for s in GEMM_COEFF_SHAPES] +
                         [(1000, 4, 7168, 0), (1000, 4, 7168, 1), (40000, 1, 64, 0),
                          (300, 8, 512, 1)])
def test_gemm_rms_coeffs_equals_the_two_calls(B, n, C, iters):
    wl = WORKLOADS["tiny"].with_(B=B, n=n, C=C, bias_std=0.3, iters=iters)
    inp = make_inputs(wl, seed=21)
    X, phi, bias = dev_bf16(inp["X"]), dev_bf16(inp["phi_t"]), dev_f32(inp["bias"])
    a, b = mhc.alloc_outputs(B, n, C), mhc.alloc_outputs(B, n, C)
    mhc.mhc_gemm_rms(X, phi, B, n, C, a["Y"], a["r"], a["ws"])
    mhc.mhc_coeffs(a["Y"], a["r"], wl.alpha_pre, wl.alpha_post, wl.alpha_res, bias, wl.iters, B,
                   n, a["H_pre"], a["H_post"], a["H_res"])
    mhc.mhc_gemm_rms_coeffs(X, phi, wl.alpha_pre, wl.alpha_post, wl.alpha_res, bias, wl.iters, B,
                            n, C, b["Y"], b["r"], b["H_pre"], b["H_post"], b["H_res"], b["ws"])
    torch.cuda.synchronize()
    for k in ("Y", "r", "H_pre", "H_post", "H_res"):
        assert torch.equal(a[k], b[k]), k
    assert mhc.mhc_device_status() == mhc.MHC_OK


# shapes for the one-kernel steps 1-4a path (test hook): a ragged last tile, a
# ragged last chunk of tiles, every n from 1 to 8, a single chunk, and the
# 7B-width workload
FUSED_SHAPES = [(1000, 4, 7168), (1100, 4, 4096), (600, 8, 2048), (256, 4, 2048), (4096, 4, 4096),
                (300, 3, 2048), (257, 1, 8192), (2000, 4, 8192), (129, 3, 3072), (700, 6, 1024),
                (520, 5, 512), (900, 7, 256), (3000, 2, 1000)]


@pytest.mark.parametrize("B,n,C", FUSED_SHAPES)
def test_forward_fused_path_shapes(B, n, C):
    wl = WORKLOADS["tiny"].with_(B=B, n=n, C=C, bias_std=0.3)
    inp = make_inputs(wl, seed=6)
    out = forward_gpu(inp, wl, path="fused")
    check_forward(out, inp, wl)
    check_properties(out, wl)
    again = forward_gpu(inp, wl, path="fused")
    for k in ("Y", "r", "H_res", "F_pre", "X_next"):
        assert torch.equal(out[k], again[k]), k  # fixed-order sums: bitwise reproducible


@pytest.mark.parametrize("B,n,C", [(64, 4, 256), (1, 4, 7168), (128, 8, 1024)])
def test_forward_fused_path_rejects_one_tile(B, n, C):
    wl = WORKLOADS["tiny"].with_(B=B, n=n, C=C)
    inp = make_inputs(wl, seed=6)
    with pytest.raises(mhc.MhcError) as ei:
        forward_gpu(inp, wl, path="fused")
    assert ei.value.status == mhc.MHC_ERR_UNSUPPORTED


def test_forward_fused_path_f_pre_uses_the_written_h_pre():
    """The finisher forms H_pre of its rows for F_pre; the stored H_pre comes from the
    coefficient warp.  With X one-hot over the streams (channel c only in stream
    c mod n), F_pre[c] is the bf16 rounding of the fp32 product H_pre[c mod n]·x[c],
    bit for bit, so a finisher that used other bits would show."""
    B, n, C = 300, 4, 4096
    wl = WORKLOADS["decode1"].with_(B=B, n=n, C=C, bias_std=0.3)
    inp = make_inputs(wl, seed=9)
    x = inp["X"].reshape(B, n, C)
    keep = (np.arange(C)[None, :] % n) == np.arange(n)[:, None]
    inp["X"] = np.where(keep[None], x, np.uint16(0)).reshape(B, n * C).astype(np.uint16)
    out = forward_gpu(inp, wl, path="fused")
    Hp = host64(out["H_pre"])
    xs = f64(inp["X"]).reshape(B, n, C)[:, np.arange(C) % n, np.arange(C)]
    prod32 = (Hp[:, np.arange(C) % n] * xs).astype(np.float32)
    assert np.array_equal(host_bits(out["F_pre"]), synth.f32_to_bf16_bits(prod32))


@pytest.mark.parametrize("B,n,C", ODD_SHAPES)
@pytest.mark.parametrize("path", ["auto", "chain"])
def test_forward_odd_shapes(B, n, C, path):
    wl = WORKLOADS["tiny"].with_(B=B, n=n, C=C, bias_std=0.3)
    inp = make_inputs(wl, seed=3)
    check_forward(forward_gpu(inp, wl, path=path), inp, wl)


@pytest.mark.parametrize("name", ["tiny", "decode1", "decode128"])
def test_forward_chain_path_small_batches(name):
    """mhc_forward takes the one-launch path for these; the chain must agree with the oracle too."""
    wl = WORKLOADS[name]
    inp = make_inputs(wl, seed=0)
    out = forward_gpu(inp, wl, path="chain")
    check_forward(out, inp, wl)
    check_properties(out, wl)


# shapes for the small-batch one-launch path: every n, ragged K blocks, ragged
# and several token tiles (up to 2048 of its 4096-token limit), one CTA and all SMs
DECODE_SHAPES = ODD_SHAPES + [(1, 4, 7168), (1, 8, 7168), (128, 4, 7168), (129, 4, 7168),
                              (300, 8, 512), (512, 4, 7168), (77, 6, 1000), (1100, 4, 2048),
                              (2048, 4, 512), (2000, 8, 264)]


@pytest.mark.parametrize("B,n,C", DECODE_SHAPES)
def test_forward_decode_path_shapes(B, n, C):
    wl = WORKLOADS["tiny"].with_(B=B, n=n, C=C, bias_std=0.3)
    inp = make_inputs(wl, seed=8)
    out = forward_gpu(inp, wl, path="decode")
    check_forward(out, inp, wl)
    check_properties(out, wl)
    again = forward_gpu(inp, wl, path="decode")
    for k in ("Y", "r", "H_pre", "H_post", "H_res", "F_pre", "X_next"):
        assert torch.equal(out[k], again[k]), k  # fixed-order sums: bitwise reproducible


def test_forward_decode_path_f_pre_uses_the_written_h_pre():
    """Every CTA that mixes a token's channels must form the same H_pre bits as the
    CTA that stores it.  With X one-hot over the streams (channel c lives in
    stream c mod n only), F_pre[c] is the bf16 rounding of the fp32 product
    H_pre[c mod n]·x[c], bit for bit, so a CTA that used other bits would show."""
    B, n, C = 3, 4, 7168  # each token's channels are spread over ~50 CTAs
    wl = WORKLOADS["decode1"].with_(B=B, n=n, C=C, bias_std=0.3)
    inp = make_inputs(wl, seed=9)
    x = inp["X"].reshape(B, n, C)
    keep = (np.arange(C)[None, :] % n) == np.arange(n)[:, None]  # [n][C]
    inp["X"] = np.where(keep[None], x, np.uint16(0)).reshape(B, n * C).astype(np.uint16)
    out = forward_gpu(inp, wl, path="decode")
    Hp = host64(out["H_pre"])  # exact fp32 values
    xs = f64(inp["X"]).reshape(B, n, C)[:, np.arange(C) % n, np.arange(C)]
    prod32 = (Hp[:, np.arange(C) % n] * xs).astype(np.float32)  # exact product, one rounding
    want = synth.f32_to_bf16_bits(prod32)
    assert np.array_equal(host_bits(out["F_pre"]), want)


@pytest.mark.parametrize("path", ["auto", "decode"])
def test_forward_decode_in_place(path):
    wl = WORKLOADS["decode32"]
    inp = make_inputs(wl, seed=4)
    ref_out = forward_gpu(inp, wl, path=path)
    out = forward_gpu(inp, wl, inplace=True, path=path)
    assert torch.equal(out["X_next"], ref_out["X_next"])
    check_forward(out, inp, wl)


def test_forward_decode_path_rejects_large_batches():
    wl = WORKLOADS["tiny"].with_(B=4097)
    inp = make_inputs(wl, seed=6)
    with pytest.raises(mhc.MhcError) as ei:
        forward_gpu(inp, wl, path="decode")
    assert ei.value.status == mhc.MHC_ERR_UNSUPPORTED


def test_sinkhorn_reciprocal_within_one_ulp():
    """The reciprocal of the Sinkhorn steps and the sigmoids (the hardware's
    approximate one): within one ulp of 1/x (fp64) wherever x and 1/x are normal
    fp32 numbers, both signs; the row and column sums it sees lie in [1, 8]."""
    rng = np.random.default_rng(5)
    mags = 10.0 ** rng.uniform(-37, 37, 200000)
    x = np.concatenate([mags * rng.choice([-1.0, 1.0], mags.size),
                        rng.uniform(1.0, 8.0, 100000),
                        2.0 ** np.arange(-120, 121)]).astype(np.float32)
    xd = torch.from_numpy(x).cuda()
    out = torch.empty_like(xd)
    mhc.mhc_testing_recip(xd, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    exact = 1.0 / x.astype(np.float64)
    ulp = np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64)
    err = np.abs(got - exact) / ulp
    assert float(err.max()) <= 1.0, float(err.max())
