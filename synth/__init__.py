"""Seeded synthetic inputs for the mHC forward workloads.

Random-number generation only: this package holds none of the mHC arithmetic.
The fp64 oracle (``oracle/``) and the CUDA path both consume the arrays made
here, so they always see identical inputs.  The generator is counter based
(splitmix64 output function + Box–Muller, see ``synth.c``): element ``i`` of
tensor ``tid`` under ``seed`` is the same whatever the array size or thread
count, so the first ``S`` rows of a workload can be generated on their own.

bf16 tensors are returned as ``numpy.uint16`` arrays holding the bf16 bit
patterns; ``bf16_bits_to_f32`` widens them exactly.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .configs import WORKLOADS, Workload, make_inputs  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_SO = os.path.join(_HERE, "_build", "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``_build/libsynth.so`` (host code, gcc)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        os.makedirs(os.path.dirname(_SO), exist_ok=True)
        tmp = _SO + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-shared", "-fPIC", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, u64, u32, i32, dbl = (ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32,
                                       ctypes.c_int, ctypes.c_double)
            vp = ctypes.c_void_p
            lib.synth_normal_bf16.argtypes = [vp, i64, u64, u32, dbl, i32]
            lib.synth_normal_f32.argtypes = [vp, i64, u64, u32, dbl, i32]
            lib.synth_rowscale_normal_bf16.argtypes = [vp, i64, i64, u64, u32, u32, dbl, dbl, i32]
            lib.synth_student_t_bf16.argtypes = [vp, i64, u64, u32, i32, dbl, i32]
            lib.synth_int_bf16.argtypes = [vp, i64, u64, u32, i32, i32, i32]
            for f in (lib.synth_normal_bf16, lib.synth_normal_f32, lib.synth_rowscale_normal_bf16,
                      lib.synth_student_t_bf16, lib.synth_int_bf16):
                f.restype = None
            _lib = lib
    return _lib


def _shape(shape):
    return (shape,) if isinstance(shape, int) else tuple(shape)


def normal_bf16(shape, seed: int, tid: int, std: float = 1.0, nthreads: int = 0) -> np.ndarray:
    out = np.empty(_shape(shape), dtype=np.uint16)
    _load().synth_normal_bf16(out.ctypes.data, out.size, seed, tid, std, nthreads)
    return out


def normal_f32(shape, seed: int, tid: int, std: float = 1.0, nthreads: int = 0) -> np.ndarray:
    out = np.empty(_shape(shape), dtype=np.float32)
    _load().synth_normal_f32(out.ctypes.data, out.size, seed, tid, std, nthreads)
    return out


def rowscale_normal_bf16(rows: int, cols: int, seed: int, tid: int, sigma_tid: int,
                         log10_lo: float = -1.0, log10_hi: float = 1.0,
                         nthreads: int = 0) -> np.ndarray:
    """Row r ~ N(0, s_r^2) with s_r = 10**U(log10_lo, log10_hi) drawn per row."""
    out = np.empty((rows, cols), dtype=np.uint16)
    _load().synth_rowscale_normal_bf16(out.ctypes.data, rows, cols, seed, tid, sigma_tid,
                                       log10_lo, log10_hi, nthreads)
    return out


def student_t_bf16(shape, seed: int, tid: int, nu: int = 3, scale: float = 1.0,
                   nthreads: int = 0) -> np.ndarray:
    """Student-t with ``nu`` degrees of freedom: Z / sqrt(chi2_nu / nu)."""
    out = np.empty(_shape(shape), dtype=np.uint16)
    _load().synth_student_t_bf16(out.ctypes.data, out.size, seed, tid, nu, scale, nthreads)
    return out


def int_bf16(shape, seed: int, tid: int, lo: int, hi: int, nthreads: int = 0) -> np.ndarray:
    """Integers uniform on [lo, hi] (exact in bf16 for |v| <= 256)."""
    out = np.empty(_shape(shape), dtype=np.uint16)
    _load().synth_int_bf16(out.ctypes.data, out.size, seed, tid, lo, hi, nthreads)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.ascontiguousarray(bits).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (NaN kept quiet)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = (u & 0x7F800000) == 0x7F800000
    nan &= (u & 0x007FFFFF) != 0
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r[nan] = ((u[nan] >> 16) | 0x40).astype(np.uint16)
    return r


# ---------------------------------------------------------------- fp8 e4m3
# OCP 8-bit floating point E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits;
# no infinities, S.1111.111 is NaN, largest finite 448, subnormals m·2^-9.


def _e4m3_table() -> np.ndarray:
    v = np.empty(256, dtype=np.float64)
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 0xF, c & 7
        if e == 15 and m == 7:
            v[c] = np.nan
        elif e == 0:
            v[c] = s * m * 2.0 ** -9
        else:
            v[c] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return v


_E4M3 = _e4m3_table()


def e4m3_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact decoding of e4m3 codes (uint8) to float32."""
    return _E4M3[np.ascontiguousarray(bits, dtype=np.uint8)].astype(np.float32)


def f32_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> e4m3 codes: round to nearest, ties to even; finite values past
    448 saturate to ±448; NaN -> 0x7F (the conversion PTX calls rn.satfinite)."""
    x = np.ascontiguousarray(x, dtype=np.float32).astype(np.float64)
    a = np.abs(x)
    sign = np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    code = np.zeros(x.shape, dtype=np.int64)
    sub = a < 2.0 ** -6
    q = np.rint(a[sub] / 2.0 ** -9).astype(np.int64)  # 8 -> the smallest normal, code 8
    code[sub] = q
    nrm = ~sub & np.isfinite(a)
    mant, ex = np.frexp(a[nrm])  # a = mant·2^ex, mant in [0.5, 1)
    e = ex - 1                   # a = (2·mant)·2^e, 2·mant in [1, 2)
    mq = np.rint((2.0 * mant - 1.0) * 8.0).astype(np.int64)
    e = np.where(mq == 8, e + 1, e)
    mq = np.where(mq == 8, 0, mq)
    field = e + 7
    over = (field > 15) | ((field == 15) & (mq == 7))
    c = np.where(over, (15 << 3) | 6, (np.clip(field, 1, 15) << 3) | mq)
    code[nrm] = c
    code[~np.isfinite(a)] = np.where(np.isnan(a[~np.isfinite(a)]), 0x7F, (15 << 3) | 6)
    out = code.astype(np.uint8) | sign
    out[np.isnan(x)] = 0x7F
    return out


def normal_e4m3(shape, seed: int, tid: int, std: float = 1.0, nthreads: int = 0) -> np.ndarray:
    """N(0, std²) rounded to e4m3 codes (uint8)."""
    return f32_to_e4m3_bits(normal_f32(shape, seed, tid, std, nthreads))
