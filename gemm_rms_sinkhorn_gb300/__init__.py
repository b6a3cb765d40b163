"""Python binding of the GB300 mHC forward library (``include/mhc.h``).

Argument marshalling only: every step of the mHC forward runs in the CUDA
kernels of ``libmhc_gb300.so``.  PyTorch supplies device memory and streams.
Importing this package raises ``ImportError`` when the library has not been
built (``python gemm_rms_sinkhorn_gb300/build.py``); there is no fallback.

Functions carry the C names and take torch tensors in the layouts of
``mhc.h`` (bf16 tensors as ``torch.bfloat16``, fp32 as ``torch.float32``, all
contiguous CUDA tensors).  ``stream`` defaults to torch's current stream.
A non-zero status raises ``MhcError``.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# MHC_GB300_CHECK=1 loads the build with device index checks (-DMHC_CHECK,
# `python gemm_rms_sinkhorn_gb300/build.py --check`) instead of the default one.
CHECK_BUILD = os.environ.get("MHC_GB300_CHECK", "0") not in ("", "0")
LIB_PATH = os.path.join(_PKG, "libmhc_gb300_check.so" if CHECK_BUILD else "libmhc_gb300.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("%s is missing: build it with `python gemm_rms_sinkhorn_gb300/build.py%s` "
                      "(or __graft_entry__.build())" % (LIB_PATH, " --check" if CHECK_BUILD else ""))

_lib = ctypes.CDLL(LIB_PATH)

MHC_OK = 0
MHC_ERR_INVALID = -1
MHC_ERR_UNSUPPORTED = -2
MHC_ERR_ALIGN = -3
MHC_ERR_CUDA = -4
MHC_ERR_TIMEOUT = -5
MHC_ERR_WORKSPACE = -6
MHC_ERR_BOUNDS = -7

MHC_NOALLOC_SCRATCH_BYTES = 16 << 20  # include/mhc.h: the built-in scratch of mhc_gemm_rms_noalloc

_vp, _i64, _i32, _f32, _sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                              ctypes.c_size_t)
_SIGS = {
    "mhc_status_str": ([_i32], ctypes.c_char_p),
    "mhc_workspace_bytes": ([_i64, _i32, _i64], _sz),
    "mhc_gemm_rms": ([_vp, _vp, _i64, _i32, _i64, _vp, _vp, _vp, _sz, _vp], _i32),
    "mhc_coeffs": ([_vp, _vp, _f32, _f32, _f32, _vp, _i32, _i64, _i32, _vp, _vp, _vp, _vp], _i32),
    "mhc_gemm_rms_coeffs": ([_vp, _vp, _f32, _f32, _f32, _vp, _i32, _i64, _i32, _i64, _vp, _vp,
                             _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "mhc_pre_apply": ([_vp, _vp, _i64, _i32, _i64, _vp, _vp], _i32),
    "mhc_post_res_apply": ([_vp, _vp, _vp, _vp, _i64, _i32, _i64, _vp, _vp], _i32),
    "mhc_forward": ([_vp, _vp, _vp, _f32, _f32, _f32, _vp, _i32, _i64, _i32, _i64,
                     _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "mhc_device_status": ([ctypes.POINTER(_i32)], _i32),
    "mhc_forward_host_scratch_bytes": ([_i64, _i32, _i64], _sz),
    "mhc_rmsnorm_gemm_workspace_bytes": ([_i64, _i64, _i64], _sz),
    "mhc_split_phi": ([_vp, _i32, _i64, _vp, _vp], _i32),
    "mhc_gemm_rms_e4m3": ([_vp, _vp, _i64, _i32, _i64, _vp, _vp, _vp, _sz, _vp], _i32),
    "mhc_pre_apply_e4m3": ([_vp, _vp, _i64, _i32, _i64, _vp, _vp], _i32),
    "mhc_post_res_apply_e4m3": ([_vp, _vp, _vp, _vp, _i64, _i32, _i64, _vp, _vp], _i32),
    "mhc_forward_e4m3": ([_vp, _vp, _vp, _f32, _f32, _f32, _vp, _i32, _i64, _i32, _i64,
                          _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "mhc_gemm_rms_split": ([_vp, _vp, _i64, _i32, _i64, _vp, _vp, _vp, _sz, _vp], _i32),
    "mhc_post_res_apply_f32": ([_vp, _vp, _vp, _vp, _i64, _i32, _i64, _vp, _vp], _i32),
    "mhc_forward_f32w": ([_vp, _vp, _vp, _f32, _f32, _f32, _vp, _i32, _i64, _i32, _i64,
                          _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "mhc_rmsnorm_gemm": ([_vp, _vp, _i64, _i64, _i64, _f32, _vp, _vp, _sz, _vp], _i32),
    "mhc_forward_host": ([_vp, _vp, _vp, _f32, _f32, _f32, _vp, _i32, _i64, _i32, _i64,
                          _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "mhc_gemm_rms_noalloc": ([_vp, _vp, _i64, _i32, _i64, _vp, _vp, _vp], _i32),
    # test hook (include/mhc_testing.h), not part of the stable API
    "mhc_testing_gemm_rms_stalled": ([_vp, _vp, _i64, _i32, _i64, _vp, _vp, _vp, _sz, _i64,
                                      ctypes.c_uint64, _vp], _i32),
    "mhc_testing_forward_fused": ([_vp, _vp, _vp, _f32, _f32, _f32, _vp, _i32, _i64, _i32, _i64,
                                   _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "mhc_testing_forward_chain": ([_vp, _vp, _vp, _f32, _f32, _f32, _vp, _i32, _i64, _i32, _i64,
                                   _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "mhc_testing_forward_decode": ([_vp, _vp, _vp, _f32, _f32, _f32, _vp, _i32, _i64, _i32,
                                    _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp],
                                   _i32),
    "mhc_testing_forward_decode_stalled": ([_vp, _vp, _vp, _f32, _f32, _f32, _vp, _i32, _i64,
                                            _i32, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                            _sz, _vp, ctypes.c_uint64], _i32),
    "mhc_testing_recip": ([_vp, _vp, _i64, _vp], _i32),
    "mhc_testing_host_chunks": ([_i64, _vp, _i64, ctypes.POINTER(_i64)], _i32),
    "mhc_testing_memory_checks": ([_i32], _i32),
    "mhc_testing_check_build": ([], _i32),
    "mhc_testing_check_record": ([ctypes.POINTER(_i32), ctypes.POINTER(_i64),
                                  ctypes.POINTER(_i64)], _i32),
    "mhc_testing_check_selftest": ([], _i32),
    "mhc_testing_forward_path": ([_i64, _i32, _i64, ctypes.POINTER(_i32)], _i32),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res

EXPORTED = tuple(_SIGS)


class MhcError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s" % (where, mhc_status_str(status)))


def mhc_status_str(status: int) -> str:
    return _lib.mhc_status_str(status).decode()


def _check(status: int, where: str) -> None:
    if status != MHC_OK:
        raise MhcError(status, where)


def _ptr(t, dtype, name):
    """Device pointer of a contiguous CUDA tensor of `dtype` (None -> NULL)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def _hptr(t, dtype, name):
    """Host pointer of a contiguous CPU tensor of `dtype`."""
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if t.is_cuda:
        raise ValueError("%s must be a host (CPU) tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def _ws(ws):
    if ws is None:
        return None, 0
    if not (isinstance(ws, torch.Tensor) and ws.is_cuda and ws.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    return ws.data_ptr(), ws.numel() * ws.element_size()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def mhc_workspace_bytes(B: int, n: int, C: int) -> int:
    return int(_lib.mhc_workspace_bytes(B, n, C))


def workspace(B: int, n: int, C: int, device=None) -> torch.Tensor:
    """A device buffer of ``mhc_workspace_bytes(B, n, C)`` bytes (at least 16)."""
    nbytes = max(16, mhc_workspace_bytes(B, n, C))
    return torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")


def mhc_gemm_rms(X, phi_t, B, n, C, Y, r, ws, stream=None):
    bf, f = torch.bfloat16, torch.float32
    p, nb = _ws(ws)
    _check(_lib.mhc_gemm_rms(_ptr(X, bf, "X"), _ptr(phi_t, bf, "phi_t"), B, n, C,
                             _ptr(Y, f, "Y"), _ptr(r, f, "r"), p, nb, _stream(stream)),
           "mhc_gemm_rms")


def mhc_coeffs(Y, r, alpha_pre, alpha_post, alpha_res, bias, iters, B, n, H_pre, H_post, H_res,
               stream=None):
    f = torch.float32
    _check(_lib.mhc_coeffs(_ptr(Y, f, "Y"), _ptr(r, f, "r"), alpha_pre, alpha_post, alpha_res,
                           _ptr(bias, f, "bias"), iters, B, n, _ptr(H_pre, f, "H_pre"),
                           _ptr(H_post, f, "H_post"), _ptr(H_res, f, "H_res"), _stream(stream)),
           "mhc_coeffs")


def mhc_gemm_rms_coeffs(X, phi_t, alpha_pre, alpha_post, alpha_res, bias, iters, B, n, C, Y, r,
                        H_pre, H_post, H_res, ws, stream=None):
    bf, f = torch.bfloat16, torch.float32
    p, nb = _ws(ws)
    _check(_lib.mhc_gemm_rms_coeffs(_ptr(X, bf, "X"), _ptr(phi_t, bf, "phi_t"), alpha_pre,
                                    alpha_post, alpha_res, _ptr(bias, f, "bias"), iters, B, n, C,
                                    _ptr(Y, f, "Y"), _ptr(r, f, "r"), _ptr(H_pre, f, "H_pre"),
                                    _ptr(H_post, f, "H_post"), _ptr(H_res, f, "H_res"), p, nb,
                                    _stream(stream)),
           "mhc_gemm_rms_coeffs")


def mhc_pre_apply(X, H_pre, B, n, C, F_pre, stream=None):
    _check(_lib.mhc_pre_apply(_ptr(X, torch.bfloat16, "X"), _ptr(H_pre, torch.float32, "H_pre"),
                              B, n, C, _ptr(F_pre, torch.bfloat16, "F_pre"), _stream(stream)),
           "mhc_pre_apply")


def mhc_post_res_apply(X, F_out, H_res, H_post, B, n, C, X_next, stream=None):
    bf, f = torch.bfloat16, torch.float32
    _check(_lib.mhc_post_res_apply(_ptr(X, bf, "X"), _ptr(F_out, bf, "F_out"),
                                   _ptr(H_res, f, "H_res"), _ptr(H_post, f, "H_post"), B, n, C,
                                   _ptr(X_next, bf, "X_next"), _stream(stream)),
           "mhc_post_res_apply")


def _forward_like(name, X, phi_t, F_out, alpha_pre, alpha_post, alpha_res, bias, iters, B, n, C,
                  Y, r, H_pre, H_post, H_res, F_pre, X_next, ws, stream, *extra):
    bf, f = torch.bfloat16, torch.float32
    p, nb = _ws(ws)
    _check(getattr(_lib, name)(
        _ptr(X, bf, "X"), _ptr(phi_t, bf, "phi_t"), _ptr(F_out, bf, "F_out"), alpha_pre,
        alpha_post, alpha_res, _ptr(bias, f, "bias"), iters, B, n, C, _ptr(Y, f, "Y"),
        _ptr(r, f, "r"), _ptr(H_pre, f, "H_pre"), _ptr(H_post, f, "H_post"),
        _ptr(H_res, f, "H_res"), _ptr(F_pre, bf, "F_pre"), _ptr(X_next, bf, "X_next"), p, nb,
        _stream(stream), *extra), name)


def mhc_forward(X, phi_t, F_out, alpha_pre, alpha_post, alpha_res, bias, iters, B, n, C,
                Y, r, H_pre, H_post, H_res, F_pre, X_next, ws, stream=None):
    _forward_like("mhc_forward", X, phi_t, F_out, alpha_pre, alpha_post, alpha_res, bias, iters,
                  B, n, C, Y, r, H_pre, H_post, H_res, F_pre, X_next, ws, stream)


def mhc_testing_forward_fused(X, phi_t, F_out, alpha_pre, alpha_post, alpha_res, bias, iters, B,
                              n, C, Y, r, H_pre, H_post, H_res, F_pre, X_next, ws, stream=None):
    """Test hook: mhc_forward through the one-kernel steps 1-4a path for large batches."""
    _forward_like("mhc_testing_forward_fused", X, phi_t, F_out, alpha_pre, alpha_post, alpha_res,
                  bias, iters, B, n, C, Y, r, H_pre, H_post, H_res, F_pre, X_next, ws, stream)


def mhc_testing_forward_chain(X, phi_t, F_out, alpha_pre, alpha_post, alpha_res, bias, iters, B,
                              n, C, Y, r, H_pre, H_post, H_res, F_pre, X_next, ws, stream=None):
    """Test hook: mhc_forward through the kernel chain (GEMM with the coefficients, pre
    apply, X_next) whatever the batch."""
    _forward_like("mhc_testing_forward_chain", X, phi_t, F_out, alpha_pre, alpha_post, alpha_res,
                  bias, iters, B, n, C, Y, r, H_pre, H_post, H_res, F_pre, X_next, ws, stream)


def mhc_testing_forward_decode(X, phi_t, F_out, alpha_pre, alpha_post, alpha_res, bias, iters,
                               B, n, C, Y, r, H_pre, H_post, H_res, F_pre, X_next, ws,
                               stream=None):
    """Test hook: mhc_forward through the small-batch one-launch path (B <= 4096)."""
    _forward_like("mhc_testing_forward_decode", X, phi_t, F_out, alpha_pre, alpha_post,
                  alpha_res, bias, iters, B, n, C, Y, r, H_pre, H_post, H_res, F_pre, X_next, ws,
                  stream)


def mhc_testing_forward_decode_stalled(X, phi_t, F_out, alpha_pre, alpha_post, alpha_res, bias,
                                       iters, B, n, C, Y, r, H_pre, H_post, H_res, F_pre, X_next,
                                       ws, wait_limit_ns, stream=None):
    """Test hook: the small-batch path with a grid barrier that never completes."""
    _forward_like("mhc_testing_forward_decode_stalled", X, phi_t, F_out, alpha_pre, alpha_post,
                  alpha_res, bias, iters, B, n, C, Y, r, H_pre, H_post, H_res, F_pre, X_next, ws,
                  stream, wait_limit_ns)


def mhc_testing_recip(x, out, stream=None):
    """Test hook: the reciprocal the Sinkhorn normalisations and sigmoids use, of each x."""
    f = torch.float32
    _check(_lib.mhc_testing_recip(_ptr(x, f, "x"), _ptr(out, f, "out"), x.numel(),
                                  _stream(stream)), "mhc_testing_recip")


def mhc_testing_host_chunks(B: int) -> list:
    """Token counts of the chunks mhc_forward_host cuts a batch of B tokens into."""
    count = ctypes.c_int64(0)
    _check(_lib.mhc_testing_host_chunks(B, None, 0, ctypes.byref(count)),
           "mhc_testing_host_chunks")
    sizes = (ctypes.c_int64 * max(count.value, 1))()
    _check(_lib.mhc_testing_host_chunks(B, sizes, count.value, ctypes.byref(count)),
           "mhc_testing_host_chunks")
    return list(sizes[:count.value])


def mhc_forward_host(X, phi_t, F_out, alpha_pre, alpha_post, alpha_res, bias, iters, B, n, C,
                     Y, r, H_pre, H_post, H_res, F_pre, X_next, scratch, stream=None):
    """mhc_forward over host tensors (X, F_out in; Y ... X_next out; page-locked for
    overlap) with device-resident phi_t and bias and a device ``scratch`` of
    ``host_scratch(B, n, C)``.  Stream-ordered: synchronise before reading outputs."""
    bf, f = torch.bfloat16, torch.float32
    p, nb = _ws(scratch)
    _check(_lib.mhc_forward_host(
        _hptr(X, bf, "X"), _ptr(phi_t, bf, "phi_t"), _hptr(F_out, bf, "F_out"), alpha_pre,
        alpha_post, alpha_res, _ptr(bias, f, "bias"), iters, B, n, C, _hptr(Y, f, "Y"),
        _hptr(r, f, "r"), _hptr(H_pre, f, "H_pre"), _hptr(H_post, f, "H_post"),
        _hptr(H_res, f, "H_res"), _hptr(F_pre, bf, "F_pre"), _hptr(X_next, bf, "X_next"), p,
        nb, _stream(stream)), "mhc_forward_host")


def _ptr8(t, name):
    """Device pointer of a contiguous CUDA tensor of e4m3 codes (uint8 or float8_e4m3fn)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype not in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        raise TypeError("%s must be uint8 or float8_e4m3fn, got %s" % (name, t.dtype))
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA tensor" % name)
    return t.data_ptr()


def mhc_gemm_rms_e4m3(X, phi_t, B, n, C, Y, r, ws, stream=None):
    f = torch.float32
    p, nb = _ws(ws)
    _check(_lib.mhc_gemm_rms_e4m3(_ptr8(X, "X"), _ptr8(phi_t, "phi_t"), B, n, C,
                                  _ptr(Y, f, "Y"), _ptr(r, f, "r"), p, nb, _stream(stream)),
           "mhc_gemm_rms_e4m3")


def mhc_pre_apply_e4m3(X, H_pre, B, n, C, F_pre, stream=None):
    _check(_lib.mhc_pre_apply_e4m3(_ptr8(X, "X"), _ptr(H_pre, torch.float32, "H_pre"), B, n, C,
                                   _ptr8(F_pre, "F_pre"), _stream(stream)), "mhc_pre_apply_e4m3")


def mhc_post_res_apply_e4m3(X, F_out, H_res, H_post, B, n, C, X_next, stream=None):
    f = torch.float32
    _check(_lib.mhc_post_res_apply_e4m3(_ptr8(X, "X"), _ptr8(F_out, "F_out"),
                                        _ptr(H_res, f, "H_res"), _ptr(H_post, f, "H_post"), B, n,
                                        C, _ptr8(X_next, "X_next"), _stream(stream)),
           "mhc_post_res_apply_e4m3")


def mhc_forward_e4m3(X, phi_t, F_out, alpha_pre, alpha_post, alpha_res, bias, iters, B, n, C,
                     Y, r, H_pre, H_post, H_res, F_pre, X_next, ws, stream=None):
    """The fp8 forward: X, phi_t, F_out, F_pre, X_next as e4m3 codes."""
    f = torch.float32
    p, nb = _ws(ws)
    _check(_lib.mhc_forward_e4m3(
        _ptr8(X, "X"), _ptr8(phi_t, "phi_t"), _ptr8(F_out, "F_out"), alpha_pre, alpha_post,
        alpha_res, _ptr(bias, f, "bias"), iters, B, n, C, _ptr(Y, f, "Y"), _ptr(r, f, "r"),
        _ptr(H_pre, f, "H_pre"), _ptr(H_post, f, "H_post"), _ptr(H_res, f, "H_res"),
        _ptr8(F_pre, "F_pre"), _ptr8(X_next, "X_next"), p, nb, _stream(stream)),
        "mhc_forward_e4m3")


def mhc_split_phi(phi_t, n, C, phi_split, stream=None):
    """fp32 phi_t [N, K] -> bf16 phi_split [2N, K] (hi, remainder interleaved)."""
    _check(_lib.mhc_split_phi(_ptr(phi_t, torch.float32, "phi_t"), n, C,
                              _ptr(phi_split, torch.bfloat16, "phi_split"), _stream(stream)),
           "mhc_split_phi")


def mhc_gemm_rms_split(X, phi_split, B, n, C, Y, r, ws, stream=None):
    bf, f = torch.bfloat16, torch.float32
    p, nb = _ws(ws)
    _check(_lib.mhc_gemm_rms_split(_ptr(X, bf, "X"), _ptr(phi_split, bf, "phi_split"), B, n, C,
                                   _ptr(Y, f, "Y"), _ptr(r, f, "r"), p, nb, _stream(stream)),
           "mhc_gemm_rms_split")


def mhc_post_res_apply_f32(X, F_out, H_res, H_post, B, n, C, X_next, stream=None):
    bf, f = torch.bfloat16, torch.float32
    _check(_lib.mhc_post_res_apply_f32(_ptr(X, bf, "X"), _ptr(F_out, f, "F_out"),
                                       _ptr(H_res, f, "H_res"), _ptr(H_post, f, "H_post"), B, n,
                                       C, _ptr(X_next, bf, "X_next"), _stream(stream)),
           "mhc_post_res_apply_f32")


def mhc_forward_f32w(X, phi_split, F_out, alpha_pre, alpha_post, alpha_res, bias, iters, B, n, C,
                     Y, r, H_pre, H_post, H_res, F_pre, X_next, ws, stream=None):
    """The fp32-weight forward: phi_split from mhc_split_phi, F_out fp32 [B, C]."""
    bf, f = torch.bfloat16, torch.float32
    p, nb = _ws(ws)
    _check(_lib.mhc_forward_f32w(
        _ptr(X, bf, "X"), _ptr(phi_split, bf, "phi_split"), _ptr(F_out, f, "F_out"), alpha_pre,
        alpha_post, alpha_res, _ptr(bias, f, "bias"), iters, B, n, C, _ptr(Y, f, "Y"),
        _ptr(r, f, "r"), _ptr(H_pre, f, "H_pre"), _ptr(H_post, f, "H_post"),
        _ptr(H_res, f, "H_res"), _ptr(F_pre, bf, "F_pre"), _ptr(X_next, bf, "X_next"), p, nb,
        _stream(stream)), "mhc_forward_f32w")


def mhc_rmsnorm_gemm(A, B_t, M, K, N, eps, C, ws=None, stream=None):
    """C = rmsnorm(A) @ B (Lazy Pre-Norm): A [M, K], B_t [N, K], C [M, N], all bf16."""
    bf = torch.bfloat16
    p, nb = _ws(ws)
    _check(_lib.mhc_rmsnorm_gemm(_ptr(A, bf, "A"), _ptr(B_t, bf, "B_t"), M, K, N, eps,
                                 _ptr(C, bf, "C"), p, nb, _stream(stream)), "mhc_rmsnorm_gemm")


def rmsnorm_gemm(A, B_t, eps: float = 1e-5, out=None, ws=None, stream=None):
    """``mhc_rmsnorm_gemm`` on tensors; allocates C and the workspace when not given."""
    M, K = A.shape
    N = B_t.shape[0]
    C = out if out is not None else torch.empty(M, N, dtype=torch.bfloat16, device=A.device)
    if ws is None:
        nbytes = _lib.mhc_rmsnorm_gemm_workspace_bytes(M, K, N)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=A.device) if nbytes else None
    mhc_rmsnorm_gemm(A, B_t, M, K, N, eps, C, ws, stream)
    return C


def host_scratch(B: int, n: int, C: int, device=None) -> "torch.Tensor":
    """Device scratch of ``mhc_forward_host`` for (B, n, C)."""
    nbytes = _lib.mhc_forward_host_scratch_bytes(B, n, C)
    if nbytes == 0 and B > 0:
        raise MhcError(MHC_ERR_INVALID, "mhc_forward_host_scratch_bytes")
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device or "cuda")


def alloc_host_outputs(B: int, n: int, C: int, pin: bool = True) -> dict:
    """Host output buffers of ``mhc_forward_host`` (page-locked when ``pin``)."""
    N = n * n + 2 * n
    f, bf = torch.float32, torch.bfloat16
    mk = lambda *shape, dtype=f: torch.empty(*shape, dtype=dtype, pin_memory=pin)
    return dict(Y=mk(B, N), r=mk(B), H_pre=mk(B, n), H_post=mk(B, n), H_res=mk(B, n, n),
                F_pre=mk(B, C, dtype=bf), X_next=mk(B, n * C, dtype=bf))


def mhc_gemm_rms_noalloc(X, phi_t, B, n, C, Y, r, stream=None):
    """mhc_gemm_rms with the library's built-in scratch: for callers that cannot
    allocate device memory (no workspace argument; calls on one device must not
    overlap on the GPU)."""
    bf, f = torch.bfloat16, torch.float32
    _check(_lib.mhc_gemm_rms_noalloc(_ptr(X, bf, "X"), _ptr(phi_t, bf, "phi_t"), B, n, C,
                                     _ptr(Y, f, "Y"), _ptr(r, f, "r"), _stream(stream)),
           "mhc_gemm_rms_noalloc")


def mhc_device_status() -> int:
    st = _i32(0)
    _check(_lib.mhc_device_status(ctypes.byref(st)), "mhc_device_status")
    return st.value


def mhc_testing_forward_path(B: int, n: int, C: int) -> str:
    """The path mhc_forward takes for (B, n, C): "decode" (one launch for steps
    1-4a) or "chain"; host-side logic only."""
    p = _i32(0)
    _check(_lib.mhc_testing_forward_path(B, n, C, ctypes.byref(p)), "mhc_testing_forward_path")
    return "decode" if p.value == 1 else "chain"


def mhc_testing_check_record() -> tuple:
    """(site, offset, extent) of the first failed device index check since the
    last read (site 0: none), read and cleared; always (0, 0, 0) in the default build."""
    site, off, ext = _i32(0), _i64(0), _i64(0)
    _check(_lib.mhc_testing_check_record(ctypes.byref(site), ctypes.byref(off), ctypes.byref(ext)),
           "mhc_testing_check_record")
    return site.value, off.value, ext.value


def alloc_outputs(B: int, n: int, C: int, device=None) -> dict:
    """Output buffers of ``mhc_forward`` for (B, n, C) plus its workspace."""
    dev = device or "cuda"
    N = n * n + 2 * n
    f, bf = torch.float32, torch.bfloat16
    return dict(Y=torch.empty(B, N, dtype=f, device=dev), r=torch.empty(B, dtype=f, device=dev),
                H_pre=torch.empty(B, n, dtype=f, device=dev),
                H_post=torch.empty(B, n, dtype=f, device=dev),
                H_res=torch.empty(B, n, n, dtype=f, device=dev),
                F_pre=torch.empty(B, C, dtype=bf, device=dev),
                X_next=torch.empty(B, n * C, dtype=bf, device=dev),
                ws=workspace(B, n, C, dev))


def forward(X, phi_t, F_out, alpha_pre, alpha_post, alpha_res, bias, iters, n, C, out=None,
            stream=None) -> dict:
    """``mhc_forward`` on tensors; allocates outputs when ``out`` is None."""
    B = X.shape[0]
    o = out if out is not None else alloc_outputs(B, n, C, X.device)
    mhc_forward(X, phi_t, F_out, alpha_pre, alpha_post, alpha_res, bias, iters, B, n, C,
                o["Y"], o["r"], o["H_pre"], o["H_post"], o["H_res"], o["F_pre"], o["X_next"],
                o["ws"], stream)
    return o
