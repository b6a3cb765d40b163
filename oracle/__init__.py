"""fp64 CPU oracle of the mHC forward pass — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
CUDA library never does, and this package imports nothing from it.

The arithmetic lives in ``mhc_oracle.c`` (plain C, double precision, one
thread, index-order sums), a restatement of §2.1–§2.5 of the page
"mHC 算法分析 & cutile 高效实现", plus C = rmsnorm(A) @ B of §2 of the page
"Towards Free Normalization: Fusing Normalization into GEMM and Attention
Kernels" (``rmsnorm_gemm``).  This module only marshals numpy arrays.

Pins: every function here is checked in ``tests/test_oracle_pins.py`` (the
pins themselves are in ``tests/oracle_pins.py``) against hand-derived worked
examples, closed forms, Sinkhorn invariants, one-hot special cases and
exact-integer results; ``tests/test_oracle_mutants.py`` plants 26 one-line
mistakes in a copy of the C source and checks that pins catch each.  No
function is left unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mhc_oracle.c")
_HDR = os.path.join(_HERE, "mhc_oracle.h")
_SO = os.path.join(_HERE, "_build", "libmhc_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (strict IEEE double: no fast-math, no FMA contraction)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < newest:
        os.makedirs(os.path.dirname(_SO), exist_ok=True)
        tmp = _SO + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-shared", "-fPIC",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _configure(lib):
    """Declare the C signatures on a loaded oracle library."""
    vp, i64, i32, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f64.restype = dbl
    lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_f64.restype = dbl
    sig = {
        "oracle_gemm_rms": [vp, vp, i64, i32, i64, vp, vp],
        "oracle_scale_bias": [vp, vp, dbl, dbl, dbl, vp, i64, i32, vp],
        "oracle_sinkhorn": [vp, i32, i32, vp],
        "oracle_constraints": [vp, i32, i64, i32, vp, vp, vp],
        "oracle_coeffs": [vp, vp, dbl, dbl, dbl, vp, i32, i64, i32, vp, vp, vp],
        "oracle_pre_apply": [vp, vp, i64, i32, i64, vp],
        "oracle_post_res_apply": [vp, vp, vp, vp, i64, i32, i64, vp],
        "oracle_forward": [vp, vp, vp, i64, i32, i64, dbl, dbl, dbl, vp, i32,
                           vp, vp, vp, vp, vp, vp, vp],
        "oracle_rmsnorm_gemm": [vp, vp, i64, i64, i64, dbl, vp],
        "oracle_gemm_rms_f64phi": [vp, vp, i64, i32, i64, vp, vp],
        "oracle_post_res_apply_f64F": [vp, vp, vp, vp, i64, i32, i64, vp],
        "oracle_forward_f64w": [vp, vp, vp, i64, i32, i64, dbl, dbl, dbl, vp, i32,
                                vp, vp, vp, vp, vp, vp, vp],
        "oracle_forward_e4m3": [vp, vp, vp, i64, i32, i64, dbl, dbl, dbl, vp, i32,
                                vp, vp, vp, vp, vp, vp, vp],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
    return _lib


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 inputs are passed as uint16 bit patterns, got %s" % a.dtype)
    return a


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _n_of_N(N: int) -> int:
    for n in range(1, 9):
        if n * n + 2 * n == N:
            return n
    raise ValueError("N=%d is not n*n+2n for n in 1..8" % N)


def bf16_to_f64(bits) -> np.ndarray:
    lib = _load()
    b = _u16(bits)
    return np.array([lib.oracle_bf16_to_f64(int(v)) for v in b.ravel()]).reshape(b.shape)


def gemm_rms(X, phi, n: int, C: int):
    """§2.1–2.2.  X [B, n*C] bf16 bits, phi [n*C, N] bf16 bits -> (Y [B,N], r [B])."""
    X, phi = _u16(X), _u16(phi)
    K = n * C
    N = n * n + 2 * n
    B = X.size // K if K else 0
    assert X.size == B * K and phi.shape == (K, N), (X.shape, phi.shape, K, N)
    Y = np.zeros((B, N))
    r = np.zeros(B)
    _load().oracle_gemm_rms(X.ctypes.data, phi.ctypes.data, B, n, C, Y.ctypes.data, r.ctypes.data)
    return Y, r


def scale_bias(Y, r, a_pre, a_post, a_res, bias):
    """§2.3.  -> H̃ [B, N]."""
    Y, r, bias = _f64(Y), _f64(r), _f64(bias)
    B, N = Y.shape
    n = _n_of_N(N)
    Ht = np.zeros((B, N))
    _load().oracle_scale_bias(Y.ctypes.data, r.ctypes.data, a_pre, a_post, a_res,
                              bias.ctypes.data, B, n, Ht.ctypes.data)
    return Ht


def sinkhorn(Ht_res, iters: int):
    """§2.4 Sinkhorn–Knopp of one n×n block (or a stack [..., n, n])."""
    Ht_res = _f64(Ht_res)
    n = Ht_res.shape[-1]
    assert Ht_res.shape[-2] == n
    flat = Ht_res.reshape(-1, n, n)
    out = np.zeros_like(flat)
    lib = _load()
    for t in range(flat.shape[0]):
        src = np.ascontiguousarray(flat[t])
        dst = np.zeros((n, n))
        lib.oracle_sinkhorn(src.ctypes.data, n, iters, dst.ctypes.data)
        out[t] = dst
    return out.reshape(Ht_res.shape)


def constraints(Ht, iters: int):
    """§2.4.  H̃ [B, N] -> (H_pre [B,n], H_post [B,n], H_res [B,n,n])."""
    Ht = _f64(Ht)
    B, N = Ht.shape
    n = _n_of_N(N)
    H_pre, H_post, H_res = np.zeros((B, n)), np.zeros((B, n)), np.zeros((B, n, n))
    _load().oracle_constraints(Ht.ctypes.data, iters, B, n, H_pre.ctypes.data,
                               H_post.ctypes.data, H_res.ctypes.data)
    return H_pre, H_post, H_res


def coeffs(Y, r, a_pre, a_post, a_res, bias, iters: int):
    """§2.3 then §2.4."""
    Y, r, bias = _f64(Y), _f64(r), _f64(bias)
    B, N = Y.shape
    n = _n_of_N(N)
    H_pre, H_post, H_res = np.zeros((B, n)), np.zeros((B, n)), np.zeros((B, n, n))
    _load().oracle_coeffs(Y.ctypes.data, r.ctypes.data, a_pre, a_post, a_res, bias.ctypes.data,
                          iters, B, n, H_pre.ctypes.data, H_post.ctypes.data, H_res.ctypes.data)
    return H_pre, H_post, H_res


def pre_apply(X, H_pre, n: int, C: int):
    """§2.5 (1).  -> F_pre [B, C] (double, unrounded)."""
    X, H_pre = _u16(X), _f64(H_pre)
    B = H_pre.shape[0]
    assert X.size == B * n * C and H_pre.shape == (B, n)
    F = np.zeros((B, C))
    _load().oracle_pre_apply(X.ctypes.data, H_pre.ctypes.data, B, n, C, F.ctypes.data)
    return F


def post_res_apply(X, F_out, H_res, H_post, n: int, C: int):
    """§2.5 (3).  -> X_next [B, n*C] (double, unrounded)."""
    X, F_out, H_res, H_post = _u16(X), _u16(F_out), _f64(H_res), _f64(H_post)
    B = H_post.shape[0]
    assert X.size == B * n * C and F_out.size == B * C
    assert H_res.size == B * n * n and H_post.shape == (B, n)
    out = np.zeros((B, n * C))
    _load().oracle_post_res_apply(X.ctypes.data, F_out.ctypes.data, H_res.ctypes.data,
                                  H_post.ctypes.data, B, n, C, out.ctypes.data)
    return out


def forward(X, phi, F_out, n: int, C: int, a_pre, a_post, a_res, bias, iters: int):
    """The whole §2 forward with F_out as an input.  Returns a dict of float64 arrays."""
    X, phi, F_out, bias = _u16(X), _u16(phi), _u16(F_out), _f64(bias)
    K, N = n * C, n * n + 2 * n
    B = X.size // K if K else 0
    assert phi.shape == (K, N) and F_out.size == B * C and bias.shape == (N,)
    o = dict(Y=np.zeros((B, N)), r=np.zeros(B), H_pre=np.zeros((B, n)), H_post=np.zeros((B, n)),
             H_res=np.zeros((B, n, n)), F_pre=np.zeros((B, C)), X_next=np.zeros((B, K)))
    _load().oracle_forward(X.ctypes.data, phi.ctypes.data, F_out.ctypes.data, B, n, C,
                           a_pre, a_post, a_res, bias.ctypes.data, iters,
                           *(o[k].ctypes.data for k in ("Y", "r", "H_pre", "H_post", "H_res",
                                                          "F_pre", "X_next")))
    return o


def rmsnorm_gemm(A, Bm, eps: float = 1e-5):
    """"Towards Free Normalization" §2: C = rmsnorm(A) @ B.  A [M, K] and Bm [K, N]
    bf16 bits (B in its mathematical orientation) -> C [M, N] float64."""
    A, Bm = _u16(A), _u16(Bm)
    M, K = A.shape
    K2, N = Bm.shape
    assert K2 == K, (A.shape, Bm.shape)
    C = np.zeros((M, N))
    _load().oracle_rmsnorm_gemm(A.ctypes.data, Bm.ctypes.data, M, K, N, float(eps), C.ctypes.data)
    return C


def gemm_rms_f64phi(X, phi, n: int, C: int):
    """§2.1–2.2 with a floating-point weight: X [B, n*C] bf16 bits, phi [n*C, N] floats."""
    X, phi = _u16(X), _f64(phi)
    K, N = n * C, n * n + 2 * n
    B = X.size // K if K else 0
    assert X.size == B * K and phi.shape == (K, N), (X.shape, phi.shape)
    Y, r = np.zeros((B, N)), np.zeros(B)
    _load().oracle_gemm_rms_f64phi(X.ctypes.data, phi.ctypes.data, B, n, C, Y.ctypes.data,
                                   r.ctypes.data)
    return Y, r


def post_res_apply_f64F(X, F_out, H_res, H_post, n: int, C: int):
    """§2.5 (3) with a floating-point F_out [B, C]."""
    X, F_out, H_res, H_post = _u16(X), _f64(F_out), _f64(H_res), _f64(H_post)
    K = n * C
    B = X.size // K if K else 0
    out = np.zeros((B, K))
    _load().oracle_post_res_apply_f64F(X.ctypes.data, F_out.ctypes.data, H_res.ctypes.data,
                                       H_post.ctypes.data, B, n, C, out.ctypes.data)
    return out


def forward_f64w(X, phi, F_out, n: int, C: int, a_pre, a_post, a_res, bias, iters: int):
    """The §2 forward with φ and F_out as floating-point inputs (X bf16 bits)."""
    X, phi, F_out, bias = _u16(X), _f64(phi), _f64(F_out), _f64(bias)
    K, N = n * C, n * n + 2 * n
    B = X.size // K if K else 0
    assert phi.shape == (K, N) and F_out.size == B * C and bias.shape == (N,)
    o = dict(Y=np.zeros((B, N)), r=np.zeros(B), H_pre=np.zeros((B, n)), H_post=np.zeros((B, n)),
             H_res=np.zeros((B, n, n)), F_pre=np.zeros((B, C)), X_next=np.zeros((B, K)))
    _load().oracle_forward_f64w(X.ctypes.data, phi.ctypes.data, F_out.ctypes.data, B, n, C,
                                a_pre, a_post, a_res, bias.ctypes.data, iters,
                                *(o[k].ctypes.data for k in ("Y", "r", "H_pre", "H_post", "H_res",
                                                             "F_pre", "X_next")))
    return o


def e4m3_to_f64(codes) -> np.ndarray:
    lib = _load()
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    return np.array([lib.oracle_e4m3_to_f64(int(v)) for v in c.ravel()]).reshape(c.shape)


def forward_e4m3(X, phi, F_out, n: int, C: int, a_pre, a_post, a_res, bias, iters: int):
    """The §2 forward on e4m3 inputs: X [B, n*C], phi [n*C, N], F_out [B, C] uint8 codes."""
    X, phi, F_out = (np.ascontiguousarray(a, dtype=np.uint8) for a in (X, phi, F_out))
    bias = _f64(bias)
    K, N = n * C, n * n + 2 * n
    B = X.size // K if K else 0
    assert phi.shape == (K, N) and F_out.size == B * C and bias.shape == (N,)
    o = dict(Y=np.zeros((B, N)), r=np.zeros(B), H_pre=np.zeros((B, n)), H_post=np.zeros((B, n)),
             H_res=np.zeros((B, n, n)), F_pre=np.zeros((B, C)), X_next=np.zeros((B, K)))
    _load().oracle_forward_e4m3(X.ctypes.data, phi.ctypes.data, F_out.ctypes.data, B, n, C,
                                a_pre, a_post, a_res, bias.ctypes.data, iters,
                                *(o[k].ctypes.data for k in ("Y", "r", "H_pre", "H_post", "H_res",
                                                             "F_pre", "X_next")))
    return o
