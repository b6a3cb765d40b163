"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

Each ``pin_*`` function raises ``AssertionError`` when the oracle disagrees
with something it must reproduce: a hand-derived worked example under
``tests/golden/``, a closed form, an invariant, or a one-hot special case.
None of them retypes the oracle's own formula.  ``test_oracle_pins.py`` runs
them against the oracle; ``test_oracle_mutants.py`` runs them against copies
of the oracle with planted mistakes and checks that some pin fails for each.

Equations: page "mHC 算法分析 & cutile 高效实现", §2.1–§2.5.  The Lazy
Pre-Norm identity: page "Towards Free Normalization: Fusing Normalization
into GEMM and Attention Kernels", §2.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16(x):
    """float values that are exactly representable in bf16 -> bit patterns."""
    x = np.asarray(x, dtype=np.float32)
    bits = synth.f32_to_bf16_bits(x)
    assert np.array_equal(synth.bf16_bits_to_f32(bits), x), "value not exact in bf16"
    return bits


def _close(a, b, tol, what):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert err <= tol, "%s: max |diff| %.3e > %.1e" % (what, err, tol)


# --------------------------------------------------------------------- bf16


def pin_bf16_widening():
    """bf16 is the top half of binary32 (IEEE 754): fixed bit patterns."""
    cases = {0x3F80: 1.0, 0xC000: -2.0, 0x3F81: 1.0 + 2.0 ** -7, 0x0001: 2.0 ** -133,
             0x7F7F: 3.3895313892515355e38, 0x0000: 0.0, 0x4040: 3.0}
    got = O.bf16_to_f64(np.array(list(cases), dtype=np.uint16))
    assert np.array_equal(got, np.array(list(cases.values()))), got
    assert math.isinf(O.bf16_to_f64(np.array([0x7F80], dtype=np.uint16))[0])


# -------------------------------------------------------------- §2.1 GEMM


def pin_gemm_onehot_rows():
    """A one-hot token row e_q picks row q of φ: Ỹ[b,:] = φ[q,:] exactly."""
    n, C = 2, 12
    K, N = n * C, n * n + 2 * n
    phi = synth.int_bf16((K, N), 7, 2, -8, 8)
    qs = [0, 5, 13, K - 1]
    X = np.zeros((len(qs), K), dtype=np.uint16)
    for b, q in enumerate(qs):
        X[b, q] = 0x3F80  # 1.0
    Y, r = O.gemm_rms(X, phi, n, C)
    phif = synth.bf16_bits_to_f32(phi).astype(np.float64)
    for b, q in enumerate(qs):
        assert np.array_equal(Y[b], phif[q]), (b, q, Y[b], phif[q])
    _close(r, np.full(len(qs), math.sqrt(1.0 / K)), 1e-15, "r of one-hot rows")


def pin_gemm_onehot_columns():
    """A one-hot column k of φ at row q_k reads X[:, q_k]: Ỹ[:,k] = X[:,q_k]."""
    n, C = 3, 8
    K, N = n * C, n * n + 2 * n
    X = synth.int_bf16((5, K), 3, 0, -100, 100)
    phi = np.zeros((K, N), dtype=np.uint16)
    picks = [(k * 7 + 3) % K for k in range(N)]
    for k, q in enumerate(picks):
        phi[q, k] = 0x3F80
    Y, _ = O.gemm_rms(X, phi, n, C)
    Xf = synth.bf16_bits_to_f32(X).astype(np.float64)
    assert np.array_equal(Y, Xf[:, picks])


def pin_gemm_integer_linearity():
    """Integer inputs give exact integer Ỹ; Ỹ is linear in X (exact below 2^53)."""
    n, C = 4, 16
    K, N = n * C, n * n + 2 * n
    X1 = synth.int_bf16((6, K), 11, 0, -2, 2)
    X2 = synth.int_bf16((6, K), 12, 0, -2, 2)
    phi = synth.int_bf16((K, N), 13, 2, -2, 2)
    Xs = _bf16(synth.bf16_bits_to_f32(X1) + synth.bf16_bits_to_f32(X2))
    Y1, _ = O.gemm_rms(X1, phi, n, C)
    Y2, _ = O.gemm_rms(X2, phi, n, C)
    Ys, _ = O.gemm_rms(Xs, phi, n, C)
    assert np.array_equal(Y1, np.round(Y1)) and np.abs(Y1).max() > 0
    assert np.array_equal(Ys, Y1 + Y2)
    # and φ scaled by -2 scales Ỹ by -2
    phi2 = _bf16(-2.0 * synth.bf16_bits_to_f32(phi))
    Y3, _ = O.gemm_rms(X1, phi2, n, C)
    assert np.array_equal(Y3, -2.0 * Y1)


# ---------------------------------------------------------------- §2.2 RMS


def pin_rms_closed_forms():
    """r = sqrt(Σx²/(nC)): a constant row s gives |s|; [3,4,0..] over K=25 gives 1."""
    n, C = 2, 8
    K, N = n * C, n * n + 2 * n
    phi = np.zeros((K, N), dtype=np.uint16)
    X = np.stack([np.full(K, v, dtype=np.float32) for v in (-3.0, 0.5, 96.0)])
    _, r = O.gemm_rms(_bf16(X), phi, n, C)
    _close(r, [3.0, 0.5, 96.0], 1e-14, "r of constant rows")
    # the divisor is K = n*C, not C: one entry 2 over K=16 gives sqrt(4/16)
    X = np.zeros((1, K), dtype=np.float32)
    X[0, 9] = 2.0
    _, r = O.gemm_rms(_bf16(X), phi, n, C)
    _close(r, [0.5], 1e-15, "r of a single spike")
    X = np.zeros((1, 25), dtype=np.float32)
    X[0, :2] = [3.0, 4.0]
    _, r = O.gemm_rms(_bf16(X), np.zeros((25, 3), dtype=np.uint16), 1, 25)
    _close(r, [1.0], 1e-15, "r of [3,4,0,...] over K=25")


# ------------------------------------------------------ §2.3 scale / bias


def pin_scale_bias_segments():
    """α = 0 gives H̃ = b; Ỹ = r·1 gives α_seg + b per column segment."""
    n = 3
    N = n * n + 2 * n
    bias = synth.normal_f32(N, 5, 3, 0.3).astype(np.float64)
    Y = synth.normal_f32((4, N), 6, 9, 2.0).astype(np.float64)
    r = np.array([0.5, 1.0, 2.0, 7.0])
    _close(O.scale_bias(Y, r, 0.0, 0.0, 0.0, bias), np.tile(bias, (4, 1)), 0.0, "α=0")
    Y1 = np.tile(r[:, None], (1, N))  # Ỹ = r, so Ỹ/r = 1
    Ht = O.scale_bias(Y1, r, 1.5, -2.0, 3.25, bias)
    want = np.concatenate([np.full(n, 1.5), np.full(n, -2.0), np.full(n * n, 3.25)]) + bias
    _close(Ht, np.tile(want, (4, 1)), 1e-15, "segment α")


def pin_lazy_prenorm_identity():
    """(A·rstd)@B = (A@B)·rstd: α·(Xφ)/r equals α·((X/r)φ), the form normalised first."""
    rng = np.random.default_rng(0)
    A = rng.standard_normal((5, 7))
    Bm = rng.standard_normal((7, 3))
    rstd = rng.uniform(0.1, 3.0, 5)
    _close((A * rstd[:, None]) @ Bm, (A @ Bm) * rstd[:, None], 1e-12, "identity")
    # the oracle's H̃ against the normalise-first form, with the rest of §2.3
    n, C = 2, 16
    K, N = n * C, n * n + 2 * n
    X = synth.normal_bf16((6, K), 21, 0, 1.0)
    phi = synth.normal_bf16((K, N), 21, 2, 0.1)
    bias = synth.normal_f32(N, 21, 3, 0.1).astype(np.float64)
    Y, r = O.gemm_rms(X, phi, n, C)
    Ht = O.scale_bias(Y, r, 0.7, 1.3, -0.4, bias)
    Xf = synth.bf16_bits_to_f32(X).astype(np.float64)
    phif = synth.bf16_bits_to_f32(phi).astype(np.float64)
    rr = np.sqrt((Xf ** 2).mean(axis=1))
    alpha = np.concatenate([np.full(n, 0.7), np.full(n, 1.3), np.full(n * n, -0.4)])
    lazy = ((Xf / rr[:, None]) @ phif) * alpha + bias
    _close(Ht, lazy, 1e-12, "H̃ vs normalise-first")


# ------------------------------------------------------ §2.4 constraints


def pin_sigmoid_points():
    g = _golden("sigmoid_points.json")
    vals = {"ln3": math.log(3.0), "-ln3": -math.log(3.0), "0": 0.0}
    n = 2
    N = n * n + 2 * n
    for p in g["points"]:
        Ht = np.zeros((1, N))
        Ht[0, :2 * n] = vals[p["Ht"]]
        H_pre, H_post, _ = O.constraints(Ht, 1)
        _close(H_pre, np.full((1, n), p["H_pre"]), 1e-15, "H_pre at " + p["Ht"])
        _close(H_post, np.full((1, n), p["H_post"]), 1e-15, "H_post at " + p["Ht"])


def pin_constraint_ranges():
    """H_pre in (0,1), H_post in (0,2), and σ(x) + σ(-x) = 1, for any input."""
    n = 4
    N = n * n + 2 * n
    Ht = synth.normal_f32((64, N), 8, 9, 6.0).astype(np.float64)
    H_pre, H_post, H_res = O.constraints(Ht, 20)
    assert (H_pre > 0).all() and (H_pre < 1).all()
    assert (H_post > 0).all() and (H_post < 2).all()
    assert (H_res > 0).all()
    H_pre_m, H_post_m, _ = O.constraints(-Ht, 20)
    _close(H_pre + H_pre_m, np.ones_like(H_pre), 1e-15, "σ(x)+σ(-x)")
    _close(H_post + H_post_m, 2 * np.ones_like(H_post), 1e-15, "2σ(x)+2σ(-x)")


def pin_sinkhorn_worked_2x2():
    g = _golden("sinkhorn_2x2.json")
    A = np.array(g["A"], dtype=np.float64)
    _close(O.sinkhorn(np.log(A), 1), g["iters1"], 1e-15, "2x2 after one iteration")
    _close(O.sinkhorn(np.log(A), 0), A, 1e-15, "iters=0 is exp(H̃)")
    p = g["limit_p"]
    _close(O.sinkhorn(np.log(A), 200), [[p, 1 - p], [1 - p, p]], 1e-12, "2x2 limit")


def pin_sinkhorn_rank_one():
    """Constant or rank-one exp(H̃) (H̃_ij = u_i + v_j) gives 1/n after one iteration."""
    for n in (1, 2, 3, 4, 8):
        _close(O.sinkhorn(np.full((n, n), 0.37), 1), np.full((n, n), 1.0 / n), 1e-15, "const")
        u = np.linspace(-2, 1, n)
        v = np.linspace(0.5, -1.5, n)
        Ht = u[:, None] + v[None, :]
        for it in (1, 2, 20):
            _close(O.sinkhorn(Ht, it), np.full((n, n), 1.0 / n), 1e-14, "rank one n=%d" % n)


def pin_sinkhorn_invariants():
    """Final step is a column step; cross-ratios are kept; row error shrinks; equivariance."""
    n = 4
    Ht = synth.normal_f32((n, n), 4, 9, 1.0).astype(np.float64)
    errs = []
    for it in range(1, 40):
        H = O.sinkhorn(Ht, it)
        _close(H.sum(axis=0), np.ones(n), 1e-12, "column sums at iters=%d" % it)
        errs.append(np.abs(H.sum(axis=1) - 1).sum())
        # cross-ratio H_ij H_kl / (H_il H_kj) = exp(H̃_ij + H̃_kl - H̃_il - H̃_kj)
        for (i, j, k, l) in ((0, 1, 2, 3), (1, 0, 3, 2), (0, 0, 1, 1)):
            cr = H[i, j] * H[k, l] / (H[i, l] * H[k, j])
            want = math.exp(Ht[i, j] + Ht[k, l] - Ht[i, l] - Ht[k, j])
            assert abs(cr / want - 1) < 1e-12, (it, cr, want)
    assert errs[0] > 1e-3, "one iteration should not already balance the rows"
    for a, b in zip(errs, errs[1:]):
        assert b <= a * (1 + 1e-9) or b < 1e-13, errs
    assert errs[-1] < 1e-10
    perm_r, perm_c = [2, 0, 3, 1], [1, 3, 0, 2]
    H = O.sinkhorn(Ht, 20)
    Hp = O.sinkhorn(Ht[perm_r][:, perm_c], 20)
    _close(Hp, H[perm_r][:, perm_c], 1e-15, "permutation equivariance")


# ---------------------------------------------------------------- §2.5 apply


def pin_pre_apply_onehot_and_half():
    """H_pre = e_i reads stream i; H_pre = 1/2 everywhere gives ½ Σ_i X[i]."""
    n, C, B = 4, 40, 3
    X = synth.normal_bf16((B, n * C), 31, 0)
    Xf = synth.bf16_bits_to_f32(X).astype(np.float64).reshape(B, n, C)
    for i in range(n):
        H = np.zeros((B, n))
        H[:, i] = 1.0
        assert np.array_equal(O.pre_apply(X, H, n, C), Xf[:, i, :])
    _close(O.pre_apply(X, np.full((B, n), 0.5), n, C), 0.5 * Xf.sum(axis=1), 1e-14, "½ΣX")


def pin_post_res_apply_permutation():
    """H_res = permutation matrix P (P[i, π(i)] = 1), H_post = 0: X_next[i] = X[π(i)]."""
    n, C, B = 3, 24, 2
    X = synth.normal_bf16((B, n * C), 32, 0)
    F = synth.normal_bf16((B, C), 32, 1)
    Xf = synth.bf16_bits_to_f32(X).astype(np.float64).reshape(B, n, C)
    pi = [1, 2, 0]  # a 3-cycle: its transpose is the other cycle
    P = np.zeros((B, n, n))
    for i in range(n):
        P[:, i, pi[i]] = 1.0
    out = O.post_res_apply(X, F, P, np.zeros((B, n)), n, C).reshape(B, n, C)
    assert np.array_equal(out, Xf[:, pi, :])


def pin_post_res_apply_post_only_and_conservation():
    """H_res = 0 gives X_next[i] = H_post[i]·F_out; column sums carry over to stream sums."""
    n, C, B = 4, 32, 3
    X = synth.normal_bf16((B, n * C), 33, 0)
    F = synth.normal_bf16((B, C), 33, 1)
    Xf = synth.bf16_bits_to_f32(X).astype(np.float64).reshape(B, n, C)
    Ff = synth.bf16_bits_to_f32(F).astype(np.float64)
    hp = np.array([[0.25, 0.5, 1.0, 2.0]] * B)
    out = O.post_res_apply(X, F, np.zeros((B, n, n)), hp, n, C).reshape(B, n, C)
    assert np.array_equal(out, hp[:, :, None] * Ff[:, None, :])
    Ht = synth.normal_f32((B, n, n), 34, 9, 1.0).astype(np.float64)
    Hres = O.sinkhorn(Ht, 20)
    out = O.post_res_apply(X, F, Hres, hp, n, C).reshape(B, n, C)
    colsum = Hres.sum(axis=1)  # [B, n]: Σ_i H_res[i, j]
    want = (colsum[:, :, None] * Xf).sum(axis=1) + hp.sum(axis=1)[:, None] * Ff
    _close(out.sum(axis=1), want, 1e-12, "stream-sum conservation")


# -------------------------------------------------------------- whole forward


def pin_forward_worked_n1():
    g = _golden("forward_n1_worked.json")
    n, C = g["n"], g["C"]
    X = _bf16(np.array([g["X"]], dtype=np.float32))
    phi = _bf16(np.array(g["phi_KxN"], dtype=np.float32))
    F = _bf16(np.array([g["F_out"]], dtype=np.float32))
    a = g["alpha"]
    o = O.forward(X, phi, F, n, C, a[0], a[1], a[2], np.array(g["bias"]), g["iters"])
    e = g["expect"]
    _close(o["Y"][0], e["Y"], 0.0, "Y")
    _close(o["r"], [e["r"]], 1e-15, "r")
    sig = lambda t: 1.0 / (1.0 + math.exp(-t))  # noqa: E731
    hp, hq = sig(e["H_pre_logit"]), 2.0 * sig(e["H_post_half_logit"])
    _close(o["H_pre"], [[hp]], 1e-15, "H_pre")
    _close(o["H_post"], [[hq]], 1e-15, "H_post")
    _close(o["H_res"][0], e["H_res"], 1e-15, "H_res")
    _close(o["F_pre"][0], hp * np.array(g["X"]), 1e-14, "F_pre")
    _close(o["X_next"][0], np.array(g["X"]) + hq * np.array(g["F_out"]), 1e-14, "X_next")


def pin_forward_alpha_zero():
    """α = 0, b = 0: H_pre = ½, H_post = 1, H_res = 1/n, so F_pre = ½ΣX[i], X_next[i] = mean X + F."""
    n, C, B = 4, 64, 5
    K, N = n * C, n * n + 2 * n
    X = synth.normal_bf16((B, K), 41, 0)
    phi = synth.normal_bf16((K, N), 41, 2, 0.02)
    F = synth.normal_bf16((B, C), 41, 1)
    o = O.forward(X, phi, F, n, C, 0.0, 0.0, 0.0, np.zeros(N), 20)
    Xf = synth.bf16_bits_to_f32(X).astype(np.float64).reshape(B, n, C)
    Ff = synth.bf16_bits_to_f32(F).astype(np.float64)
    _close(o["H_pre"], np.full((B, n), 0.5), 1e-15, "H_pre")
    _close(o["H_post"], np.ones((B, n)), 1e-15, "H_post")
    _close(o["H_res"], np.full((B, n, n), 1.0 / n), 1e-15, "H_res")
    _close(o["F_pre"], 0.5 * Xf.sum(axis=1), 1e-13, "F_pre")
    want = np.repeat(Xf.mean(axis=1, keepdims=True), n, axis=1) + Ff[:, None, :]
    _close(o["X_next"].reshape(B, n, C), want, 1e-13, "X_next")


def pin_forward_matches_steps_and_logits():
    """forward() is the composition of the steps; H̃ recovered from outputs is α(X/r)φ + b."""
    n, C, B = 2, 24, 4
    K, N = n * C, n * n + 2 * n
    X = synth.normal_bf16((B, K), 51, 0)
    phi = synth.normal_bf16((K, N), 51, 2, 0.2)
    F = synth.normal_bf16((B, C), 51, 1)
    bias = synth.normal_f32(N, 51, 3, 0.1).astype(np.float64)
    al = (0.3, -0.2, 0.5)
    o = O.forward(X, phi, F, n, C, *al, bias, 0)
    Xf = synth.bf16_bits_to_f32(X).astype(np.float64)
    phif = synth.bf16_bits_to_f32(phi).astype(np.float64)
    rr = np.sqrt((Xf ** 2).mean(axis=1))
    alpha = np.concatenate([np.full(n, al[0]), np.full(n, al[1]), np.full(n * n, al[2])])
    lazy = ((Xf / rr[:, None]) @ phif) * alpha + bias
    logit = lambda p: np.log(p) - np.log1p(-p)  # noqa: E731
    # a value outside (0, 1) or a non-positive H_res gives NaN, which fails _close
    with np.errstate(invalid="ignore", divide="ignore"):
        _close(logit(o["H_pre"]), lazy[:, :n], 1e-11, "pre logit")
        _close(logit(o["H_post"] / 2), lazy[:, n:2 * n], 1e-11, "post logit")
        _close(np.log(o["H_res"].reshape(B, n * n)), lazy[:, 2 * n:], 1e-12, "res log (iters=0)")


# ------------------------------------ "Towards Free Normalization" §2


def pin_rmsnorm_gemm_exact_rows():
    """rstd = 1/sqrt(Σa²/K + eps) on rows whose value is exact: [1,1,1,1] and
    [2,0,0,0] have mean square 1, so eps = 3 gives rstd = 1/2; with B = I the
    product is the scaled rows, exactly.  A zero row stays zero."""
    A = _bf16([[1, 1, 1, 1], [2, 0, 0, 0], [0, 0, 0, 0], [1, -1, 1, -1]])
    I4 = _bf16(np.eye(4))
    C = O.rmsnorm_gemm(A, I4, eps=3.0)
    want = np.array([[0.5, 0.5, 0.5, 0.5], [1, 0, 0, 0], [0, 0, 0, 0], [0.5, -0.5, 0.5, -0.5]])
    assert np.array_equal(C, want), C
    # eps = 0: the same rows scaled to unit mean square
    C0 = O.rmsnorm_gemm(A[[0, 1, 3]], I4, eps=0.0)
    assert np.array_equal(C0, [[1, 1, 1, 1], [2, 0, 0, 0], [1, -1, 1, -1]]), C0


def pin_rmsnorm_gemm_constant_rows():
    """A row of constant s: rstd = 1/sqrt(s² + eps), C = s·rstd·(column sums of B)."""
    K, N = 24, 5
    Bm = synth.normal_bf16((K, N), 31, 2, 0.5)
    Bf = synth.bf16_bits_to_f32(Bm).astype(np.float64)
    for s_, eps in ((0.5, 1e-5), (-3.0, 0.25), (2.0, 0.0)):
        A = _bf16(np.full((1, K), s_))
        want = s_ / math.sqrt(s_ * s_ + eps) * Bf.sum(axis=0)
        _close(O.rmsnorm_gemm(A, Bm, eps)[0], want, 1e-13, "constant row s=%g" % s_)


def pin_rmsnorm_gemm_lazy_identity():
    """The lazy order of the page's §2: with eps = 0, rmsnorm(A) @ B times r equals
    A @ B, i.e. the mHC oracle's Ỹ (n = 1, so φ is K × 3) for the same A."""
    C_, n = 40, 1
    K, N = n * C_, n * n + 2 * n
    X = synth.normal_bf16((7, K), 33, 0, 1.0)
    phi = synth.normal_bf16((K, N), 33, 2, 0.2)
    Y, r = O.gemm_rms(X, phi, n, C_)
    Cn = O.rmsnorm_gemm(X, phi, eps=0.0)
    _close(Cn * r[:, None], Y, 1e-12 * max(1.0, float(np.abs(Y).max())), "rmsnorm(A)@B · r = A@B")
    # eps > 0 shrinks every row by sqrt(r² / (r² + eps)) relative to eps = 0
    Ce = O.rmsnorm_gemm(X, phi, eps=0.3)
    _close(Ce, Cn * (r / np.sqrt(r * r + 0.3))[:, None], 1e-12, "eps scaling")


# ------------------------------- fp32 weight / fp32 F_out (the page's §5)


def pin_f64phi_and_f64F_agree_on_bf16_values():
    """φ and F_out whose values are bf16: the float-input variants equal the pinned
    bf16-input functions exactly (same values, same order)."""
    n, C_ = 3, 20
    K, N = n * C_, n * n + 2 * n
    X = synth.normal_bf16((9, K), 61, 0, 1.0)
    phi = synth.normal_bf16((K, N), 61, 2, 0.1)
    Fo = synth.normal_bf16((9, C_), 61, 1, 1.0)
    Y, r = O.gemm_rms(X, phi, n, C_)
    Y2, r2 = O.gemm_rms_f64phi(X, synth.bf16_bits_to_f32(phi), n, C_)
    assert np.array_equal(Y, Y2) and np.array_equal(r, r2)
    Hr = O.sinkhorn(synth.normal_f32((9, n, n), 61, 9, 1.0), 20)
    Hq = np.abs(synth.normal_f32((9, n), 61, 8, 0.5)).astype(np.float64)
    a = O.post_res_apply(X, Fo, Hr, Hq, n, C_)
    b = O.post_res_apply_f64F(X, synth.bf16_bits_to_f32(Fo), Hr, Hq, n, C_)
    assert np.array_equal(a, b)


def pin_f64phi_uses_the_fp32_bits():
    """Integer X and φ = φ1 + 2^-12·φ2 with small integers: Ỹ = Ỹ(φ1) + 2^-12·Ỹ(φ2)
    exactly, so the bits below bf16's mantissa count."""
    n, C_ = 2, 12
    K, N = n * C_, n * n + 2 * n
    X = synth.int_bf16((5, K), 62, 0, -3, 3)
    p1 = synth.bf16_bits_to_f32(synth.int_bf16((K, N), 62, 2, -2, 2)).astype(np.float64)
    p2 = synth.bf16_bits_to_f32(synth.int_bf16((K, N), 62, 4, -2, 2)).astype(np.float64)
    phi = (p1 + p2 * 2.0 ** -12).astype(np.float32).astype(np.float64)
    assert np.array_equal(phi, p1 + p2 * 2.0 ** -12)  # exact in fp32
    Y, _ = O.gemm_rms_f64phi(X, phi, n, C_)
    Y1, _ = O.gemm_rms_f64phi(X, p1, n, C_)
    Y2, _ = O.gemm_rms_f64phi(X, p2, n, C_)
    assert np.array_equal(Y, Y1 + Y2 * 2.0 ** -12)


def pin_f64F_post_only():
    """H_res = 0: X_next[i] = H_post[i]·F_out with F_out's full fp32 value."""
    n, C_ = 2, 8
    X = synth.normal_bf16((3, n * C_), 63, 0, 1.0)
    Fo = (synth.normal_f32((3, C_), 63, 1, 1.0) * 1.0001).astype(np.float64)
    Hq = np.array([[0.5, 2.0], [1.0, 0.25], [1.5, 0.75]])
    out = O.post_res_apply_f64F(X, Fo, np.zeros((3, n, n)), Hq, n, C_).reshape(3, n, C_)
    assert np.array_equal(out, Hq[:, :, None] * Fo[:, None, :])


# ------------------------------------------- fp8 e4m3 (the page's §4)


def pin_e4m3_decode_values():
    """Codes of the E4M3 format: 0x38 = 1, 0x7E = 448 (largest), 0x08 = 2^-6 (smallest
    normal), 0x01 = 2^-9 (smallest subnormal), 0x3C = 1.5, 0xC4 = -3, 0x7F NaN, 0x80 = -0."""
    got = O.e4m3_to_f64([0x38, 0x7E, 0x08, 0x01, 0x3C, 0xC4, 0x00, 0x07, 0x77])
    assert got.tolist() == [1.0, 448.0, 2.0 ** -6, 2.0 ** -9, 1.5, -3.0, 0.0, 7 * 2.0 ** -9, 240.0]
    assert math.isnan(O.e4m3_to_f64([0x7F])[0]) and math.isnan(O.e4m3_to_f64([0xFF])[0])
    assert math.copysign(1.0, O.e4m3_to_f64([0x80])[0]) == -1.0


def pin_forward_e4m3_equals_bf16_on_shared_values():
    """Inputs whose values are exact in both e4m3 and bf16 (multiples of 1/4 up to 3,
    0.0625·k for φ): the e4m3 forward equals the pinned bf16 forward exactly."""
    n, C_ = 3, 16
    K, N = n * C_, n * n + 2 * n
    X = synth.int_bf16((6, K), 64, 0, -12, 12)
    Fo = synth.int_bf16((6, C_), 64, 1, -12, 12)
    phi = synth.int_bf16((K, N), 64, 2, -8, 8)
    q = lambda bits, s: (synth.bf16_bits_to_f32(bits) * s).astype(np.float32)
    Xv, Fv, Pv = q(X, 0.25), q(Fo, 0.25), q(phi, 0.0625)
    bias = synth.normal_f32(N, 64, 3, 0.1).astype(np.float64)
    args = (n, C_, 0.5, 0.7, 0.9, bias, 20)
    a = O.forward(synth.f32_to_bf16_bits(Xv), synth.f32_to_bf16_bits(Pv),
                  synth.f32_to_bf16_bits(Fv), *args)
    b = O.forward_e4m3(synth.f32_to_e4m3_bits(Xv), synth.f32_to_e4m3_bits(Pv),
                       synth.f32_to_e4m3_bits(Fv), *args)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
