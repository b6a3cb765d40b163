"""The C ABI without a GPU: the library loads, exports every call that
include/mhc.h declares, and rejects bad arguments on the host before any
device work.  Pointers here are fake addresses that are never dereferenced
on a machine without a GPU: calls whose arguments pass every host check stop
at the device check there.  On a machine with a GPU those calls would launch
kernels on the fake addresses, so every test that passes them is skipped
wherever a CUDA device is visible (`no_gpu`).
"""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(os.path.join(ROOT, "include", h) for h in os.listdir(os.path.join(ROOT, "include"))
                 if h.endswith(".h"))

mhc = pytest.importorskip("gemm_rms_sinkhorn_gb300")
L = mhc._lib

import torch  # noqa: E402  (the binding has imported it already)

no_gpu = pytest.mark.skipif(torch.cuda.is_available(),
                            reason="fake device addresses: only where no GPU is visible")


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(mhc_[a-z_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_five_calls():
    names = declared_functions()
    for f in ("mhc_gemm_rms", "mhc_coeffs", "mhc_pre_apply", "mhc_post_res_apply", "mhc_forward"):
        assert f in names


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    out = subprocess.run(["nm", "-D", "--defined-only", mhc.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (mhc_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(L, n)
    assert set(names) <= set(mhc.EXPORTED)


def test_status_strings():
    for st in range(-6, 1):
        s = mhc.mhc_status_str(st)
        assert s.startswith("MHC_")
    assert "unknown" in mhc.mhc_status_str(-99)


# fake, 16-byte aligned, far-apart device addresses
A, B_, C_, D, E, F, G, H, I, J, W = [0x10000000 * (k + 1) for k in range(11)]


def gemm(X=A, phi=B_, Bt=4, n=4, C=256, Y=C_, r=D, ws=W, wsb=1 << 30):
    return L.mhc_gemm_rms(X, phi, Bt, n, C, Y, r, ws, wsb, None)


def coeffs(Y=A, r=B_, bias=C_, iters=20, Bt=4, n=4, hp=D, hq=E, hr=F):
    return L.mhc_coeffs(Y, r, 0.01, 0.01, 0.01, bias, iters, Bt, n, hp, hq, hr, None)


def gemm_coeffs(X=A, phi=B_, bias=C_, iters=20, Bt=4, n=4, C=256, Y=D, r=E, hp=F, hq=G, hr=H,
                ws=W, wsb=1 << 30):
    return L.mhc_gemm_rms_coeffs(X, phi, 0.01, 0.01, 0.01, bias, iters, Bt, n, C, Y, r, hp, hq,
                                 hr, ws, wsb, None)


def pre(X=A, Hp=B_, Bt=4, n=4, C=256, Fp=C_):
    return L.mhc_pre_apply(X, Hp, Bt, n, C, Fp, None)


def post(X=A, Fo=B_, Hr=C_, Hq=D, Bt=4, n=4, C=256, Xn=E):
    return L.mhc_post_res_apply(X, Fo, Hr, Hq, Bt, n, C, Xn, None)


def fwd(X=A, phi=B_, Fo=C_, bias=D, iters=20, Bt=4, n=4, C=256, Y=E, r=F, hp=G, hq=H, hr=I,
        Fp=J, Xn=0x1_0000_0000, ws=W, wsb=1 << 30):
    return L.mhc_forward(X, phi, Fo, 0.01, 0.01, 0.01, bias, iters, Bt, n, C, Y, r, hp, hq, hr,
                         Fp, Xn, ws, wsb, None)


NO_DEVICE = mhc.MHC_ERR_CUDA  # valid host arguments reach the device check


@no_gpu
def test_empty_batch_is_a_noop():
    assert gemm(Bt=0, X=None, phi=None, Y=None, r=None, ws=None, wsb=0) == mhc.MHC_OK
    assert coeffs(Bt=0) == mhc.MHC_OK
    assert gemm_coeffs(Bt=0) == mhc.MHC_OK
    assert pre(Bt=0) == mhc.MHC_OK
    assert post(Bt=0) == mhc.MHC_OK
    assert fwd(Bt=0) == mhc.MHC_OK


@no_gpu
@pytest.mark.parametrize("call", [gemm, gemm_coeffs, pre, post, fwd])
def test_shape_rules(call):
    assert call(n=0) == mhc.MHC_ERR_UNSUPPORTED
    assert call(n=9) == mhc.MHC_ERR_UNSUPPORTED
    assert call(C=12) == mhc.MHC_ERR_UNSUPPORTED
    assert call(C=0) == mhc.MHC_ERR_UNSUPPORTED
    assert call(Bt=-1) == mhc.MHC_ERR_INVALID
    assert call(Bt=1 << 31) == mhc.MHC_ERR_UNSUPPORTED  # token rows are 32-bit TMA coordinates


@no_gpu
def test_coeffs_rules():
    assert coeffs(n=9) == mhc.MHC_ERR_UNSUPPORTED
    assert coeffs(iters=-1) == mhc.MHC_ERR_INVALID
    assert gemm_coeffs(iters=-1) == mhc.MHC_ERR_INVALID
    assert gemm_coeffs(bias=None) == mhc.MHC_ERR_INVALID
    assert gemm_coeffs(hr=H + 4) == mhc.MHC_ERR_ALIGN
    assert gemm_coeffs(hq=A + 64) == mhc.MHC_ERR_INVALID  # an output over X
    assert gemm_coeffs(hp=G) == mhc.MHC_ERR_INVALID       # two outputs over each other
    assert gemm_coeffs() == NO_DEVICE
    assert fwd(iters=-1) == mhc.MHC_ERR_INVALID
    assert coeffs(Y=None) == mhc.MHC_ERR_INVALID


@no_gpu
def test_null_and_alignment():
    assert gemm(X=None) == mhc.MHC_ERR_INVALID
    assert pre(Fp=None) == mhc.MHC_ERR_INVALID
    assert post(Hr=None) == mhc.MHC_ERR_INVALID
    assert fwd(bias=None) == mhc.MHC_ERR_INVALID
    assert gemm(X=A + 8) == mhc.MHC_ERR_ALIGN
    assert post(Xn=E + 4) == mhc.MHC_ERR_ALIGN
    assert coeffs(hr=F + 4) == mhc.MHC_ERR_ALIGN


@no_gpu
def test_overlap_rules():
    # an output over an input
    assert gemm(Y=A + 64) == mhc.MHC_ERR_INVALID
    assert pre(Fp=A + 256) == mhc.MHC_ERR_INVALID
    # two outputs over each other
    assert coeffs(hq=D + 16) == mhc.MHC_ERR_INVALID
    # partial overlap of X_next and X is rejected, exact aliasing is accepted
    assert post(Xn=A + 1024) == mhc.MHC_ERR_INVALID
    assert post(Xn=A) == NO_DEVICE
    assert fwd(Xn=A) == NO_DEVICE
    assert fwd(Fp=A) == mhc.MHC_ERR_INVALID


@no_gpu
def test_valid_arguments_reach_the_device_check():
    assert gemm() == NO_DEVICE
    assert coeffs() == NO_DEVICE
    assert pre() == NO_DEVICE
    assert post() == NO_DEVICE
    assert fwd() == NO_DEVICE
    assert mhc.mhc_workspace_bytes(64, 4, 256) == 0  # needs a device
    assert mhc.mhc_workspace_bytes(64, 9, 256) == 0


def test_binding_fails_loudly_without_the_library(tmp_path):
    """A copy of the package without libmhc_gb300.so must not import (no fallback)."""
    import shutil
    pkg = os.path.join(ROOT, "gemm_rms_sinkhorn_gb300")
    dst = tmp_path / "gemm_rms_sinkhorn_gb300"
    shutil.copytree(pkg, dst, ignore=shutil.ignore_patterns("*.so", "_build", "__pycache__"))
    code = "import gemm_rms_sinkhorn_gb300"
    res = subprocess.run([sys.executable, "-c", code], cwd=tmp_path, capture_output=True,
                         text=True)
    assert res.returncode != 0 and "ImportError" in res.stderr


@no_gpu
def test_testing_hooks_validate_on_the_host():
    assert L.mhc_testing_recip(A, B_, -1, None) == mhc.MHC_ERR_INVALID
    assert L.mhc_testing_recip(A, B_, 0, None) == mhc.MHC_OK
    assert L.mhc_testing_recip(None, B_, 4, None) == mhc.MHC_ERR_INVALID
    assert L.mhc_testing_recip(A + 4, B_, 4, None) == mhc.MHC_ERR_ALIGN
    assert L.mhc_testing_recip(A, A + 8, 4, None) in (mhc.MHC_ERR_ALIGN, mhc.MHC_ERR_INVALID)
    assert L.mhc_testing_recip(A, B_, 4, None) == NO_DEVICE
    for name in ("mhc_testing_forward_chain", "mhc_testing_forward_decode"):
        f = getattr(L, name)
        args = [A, B_, C_, 0.01, 0.01, 0.01, D, 20, 4, 4, 256, E, F, G, H, I, J,
                0x1_0000_0000, W, 1 << 30, None]
        assert f(*args) == NO_DEVICE
        args[8] = 0
        assert f(*args) == mhc.MHC_OK  # empty batch
        args[8], args[9] = 4, 9
        assert f(*args) == mhc.MHC_ERR_UNSUPPORTED
    args = [A, B_, C_, 0.01, 0.01, 0.01, D, -1, 4, 4, 256, E, F, G, H, I, J, 0x1_0000_0000, W,
            1 << 30, None, 50_000_000]
    assert L.mhc_testing_forward_decode_stalled(*args) == mhc.MHC_ERR_INVALID


@no_gpu
def test_forward_host_validates_on_the_host():
    f = L.mhc_forward_host
    args = [A, B_, C_, 0.01, 0.01, 0.01, D, 20, 4, 4, 256, E, F, G, H, I, J, 0x1_0000_0000, W,
            1 << 30, None]
    assert f(*args) == NO_DEVICE
    a = list(args); a[8] = 0
    assert f(*a) == mhc.MHC_OK  # empty batch
    a = list(args); a[9] = 9
    assert f(*a) == mhc.MHC_ERR_UNSUPPORTED
    a = list(args); a[7] = -1
    assert f(*a) == mhc.MHC_ERR_INVALID
    a = list(args); a[0] = None
    assert f(*a) == mhc.MHC_ERR_INVALID
    a = list(args); a[18] = W + 8  # scratch misaligned
    assert f(*a) == mhc.MHC_ERR_ALIGN
    a = list(args); a[17] = A  # X_next == X is allowed
    assert f(*a) == NO_DEVICE
    a = list(args); a[16] = A  # F_pre over X is not
    assert f(*a) == mhc.MHC_ERR_INVALID
    assert mhc._lib.mhc_forward_host_scratch_bytes(64, 4, 256) == 0  # needs a device


@no_gpu
def test_rmsnorm_gemm_validates_on_the_host():
    f = L.mhc_rmsnorm_gemm
    assert f(A, B_, 0, 64, 64, 1e-5, C_, None, 0, None) == mhc.MHC_OK  # empty
    assert f(A, B_, 16, 64, 64, 1e-5, C_, W, 1 << 30, None) == NO_DEVICE
    assert f(A, B_, 16, 12, 64, 1e-5, C_, W, 1 << 30, None) == mhc.MHC_ERR_UNSUPPORTED
    assert f(A, B_, 16, 64, 20, 1e-5, C_, W, 1 << 30, None) == mhc.MHC_ERR_UNSUPPORTED
    assert f(A, B_, 16, 64, 64, -1.0, C_, W, 1 << 30, None) == mhc.MHC_ERR_INVALID
    assert f(A, B_, 16, 64, 64, float("nan"), C_, W, 1 << 30, None) == mhc.MHC_ERR_INVALID
    assert f(A, B_, -1, 64, 64, 1e-5, C_, W, 1 << 30, None) == mhc.MHC_ERR_INVALID
    assert f(A, B_, 1 << 31, 64, 64, 1e-5, C_, W, 1 << 30, None) == mhc.MHC_ERR_UNSUPPORTED
    assert f(A, B_, 16, 1 << 31, 64, 1e-5, C_, W, 1 << 30, None) == mhc.MHC_ERR_UNSUPPORTED
    assert f(None, B_, 16, 64, 64, 1e-5, C_, W, 1 << 30, None) == mhc.MHC_ERR_INVALID
    assert f(A + 8, B_, 16, 64, 64, 1e-5, C_, W, 1 << 30, None) == mhc.MHC_ERR_ALIGN
    assert f(A, B_, 16, 64, 64, 1e-5, A + 64, W, 1 << 30, None) == mhc.MHC_ERR_INVALID
    assert mhc._lib.mhc_rmsnorm_gemm_workspace_bytes(16, 64, 64) == 0  # needs a device


@no_gpu
def test_e4m3_calls_validate_on_the_host():
    assert L.mhc_pre_apply_e4m3(A, B_, 4, 4, 24, C_, None) == mhc.MHC_ERR_UNSUPPORTED  # C % 16
    assert L.mhc_pre_apply_e4m3(A, B_, 4, 4, 32, C_, None) == NO_DEVICE
    assert L.mhc_gemm_rms_e4m3(A, B_, 4, 4, 32, C_, D, W, 1 << 30, None) == NO_DEVICE
    assert L.mhc_post_res_apply_e4m3(A, B_, C_, D, 4, 4, 32, A, None) == NO_DEVICE  # in place
    assert L.mhc_post_res_apply_e4m3(A, B_, C_, D, 4, 4, 32, A + 16, None) == mhc.MHC_ERR_INVALID


@pytest.mark.parametrize("B", [1, 2, 3, 7, 100, 1000, 1023, 1024, 2000, 2559, 2560, 2561,
                               4100, 16384, 100000])
def test_host_chunk_plan(B):
    """mhc_forward_host's chunks (host logic, no device): they cover the batch in
    order, none exceeds 1024 tokens, large batches ramp 256, 512 up and 512, 256
    down around full chunks, and small ones go in equal chunks."""
    c = mhc.mhc_testing_host_chunks(B)
    assert sum(c) == B and all(v > 0 for v in c) and max(c) <= 1024
    if B >= 2560:
        assert c[:2] == [256, 512] and c[-2:] == [512, 256]
        mid = c[2:-2]
        assert all(v == 1024 for v in mid[:-1]) and 0 < mid[-1] <= 1024
    else:
        step = max(min(B, 1024) // 4, 1)
        assert all(v == step for v in c[:-1]) and 0 < c[-1] <= step


def test_host_chunk_plan_rules():
    count = ctypes.c_int64(-1)
    f = L.mhc_testing_host_chunks
    assert f(0, None, 0, ctypes.byref(count)) == mhc.MHC_OK and count.value == 0
    assert f(-1, None, 0, ctypes.byref(count)) == mhc.MHC_ERR_INVALID
    assert f(10, None, 0, None) == mhc.MHC_ERR_INVALID
    assert f(10, None, 4, ctypes.byref(count)) == mhc.MHC_ERR_INVALID
    sizes = (ctypes.c_int64 * 2)()
    assert f(16384, sizes, 2, ctypes.byref(count)) == mhc.MHC_OK  # capacity below the count
    assert count.value == 19 and list(sizes) == [256, 512]
