"""mhc_gemm_rms_noalloc: the entry point for callers that cannot allocate
device memory (for example code whose device memory is all owned by a host
framework's pool, or a latency-critical path where a cudaMalloc and the device
synchronisation it can bring are not acceptable).  It runs the same GEMM+RMS
kernel as mhc_gemm_rms with the split-K scratch in the library's built-in
device array.  These tests call it through the C ABI and compare it with
mhc_gemm_rms on the same inputs, two calls in a row, so the second call runs
on the scratch the first one left behind.

This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_util import R_REL, assert_rel, assert_Y_close, cuda_ok, dev_bf16, host64
from synth import WORKLOADS, make_inputs

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]

mhc = pytest.importorskip("gemm_rms_sinkhorn_gb300")


def _with_workspace(X, phi_t, B, n, C):
    N = n * n + 2 * n
    Y = torch.empty(B, N, dtype=torch.float32, device="cuda")
    r = torch.empty(B, dtype=torch.float32, device="cuda")
    ws = mhc.workspace(B, n, C)
    st = mhc._lib.mhc_gemm_rms(X.data_ptr(), phi_t.data_ptr(), B, n, C, Y.data_ptr(),
                               r.data_ptr(), ws.data_ptr(), ws.numel(), None)
    assert st == mhc.MHC_OK, mhc.mhc_status_str(st)
    return Y, r


def _no_alloc(X, phi_t, B, n, C):
    N = n * n + 2 * n
    Y = torch.full((B, N), float("nan"), dtype=torch.float32, device="cuda")
    r = torch.full((B,), float("nan"), dtype=torch.float32, device="cuda")
    st = mhc._lib.mhc_gemm_rms_noalloc(X.data_ptr(), phi_t.data_ptr(), B, n, C, Y.data_ptr(),
                                       r.data_ptr(), None)
    assert st == mhc.MHC_OK, mhc.mhc_status_str(st)
    return Y, r


@pytest.mark.parametrize("names", [("tiny", "decode8"), ("7b", "wider"), ("decode128", "tiny")])
def test_no_alloc_matches_workspace_call_twice_in_a_row(names):
    for name in names:
        wl = WORKLOADS[name]
        inp = make_inputs(wl, seed=5, parts=("X", "phi_t"))
        X, phi_t = dev_bf16(inp["X"]), dev_bf16(inp["phi_t"])
        Yw, rw = _with_workspace(X, phi_t, wl.B, wl.n, wl.C)
        Yn, rn = _no_alloc(X, phi_t, wl.B, wl.n, wl.C)
        torch.cuda.synchronize()
        assert_Y_close(host64(Yn), host64(Yw), inp["X"], inp["phi_t"], "Y (" + name + ")")
        assert_rel(host64(rn), host64(rw), R_REL, "r (" + name + ")")
        # same kernel and schedule: the results are in fact identical
        assert torch.equal(Yn, Yw) and torch.equal(rn, rw)


def test_no_alloc_rejects_problems_beyond_its_scratch():
    # n=8 needs more than the built-in scratch beyond B = 32,256 tokens; the
    # call is refused on the host, so these buffers are never touched
    B, n, C = 1 << 20, 8, 4096
    need = mhc.mhc_workspace_bytes(B, n, C)
    assert need > (16 << 20)
    big = torch.empty(16, dtype=torch.uint8, device="cuda")
    base = big.data_ptr()
    X, phi, Y, r = base, base + (1 << 40), base + (2 << 40), base + (3 << 40)
    st = mhc._lib.mhc_gemm_rms_noalloc(X, phi, B, n, C, Y, r, None)
    assert st == mhc.MHC_ERR_WORKSPACE


def test_no_alloc_empty_batch_and_bad_shape():
    assert mhc._lib.mhc_gemm_rms_noalloc(None, None, 0, 4, 256, None, None, None) == mhc.MHC_OK
    assert mhc._lib.mhc_gemm_rms_noalloc(None, None, 0, 9, 256, None, None, None) == \
        mhc.MHC_ERR_UNSUPPORTED
