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
    """The GEMM's split-K scratch grows with B and n, not C: at B=40000, n=8, C=8
    it exceeds the built-in 16 MiB while X is 5 MB.  Every buffer is real device
    memory, so no ordering of the host checks can send a kernel to a bad address."""
    B, n, C = 40000, 8, 8
    N, K = n * n + 2 * n, n * C
    limit = mhc.MHC_NOALLOC_SCRATCH_BYTES
    X = torch.zeros(B, K, dtype=torch.bfloat16, device="cuda")
    phi = torch.zeros(N, K, dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros(B, N, dtype=torch.float32, device="cuda")
    r = torch.zeros(B, dtype=torch.float32, device="cuda")
    ws = torch.zeros(limit, dtype=torch.uint8, device="cuda")
    # the GEMM itself refuses a workspace of exactly the built-in size: its need is larger
    st = mhc._lib.mhc_gemm_rms(X.data_ptr(), phi.data_ptr(), B, n, C, Y.data_ptr(),
                               r.data_ptr(), ws.data_ptr(), limit, None)
    assert st == mhc.MHC_ERR_WORKSPACE
    st = mhc._lib.mhc_gemm_rms_noalloc(X.data_ptr(), phi.data_ptr(), B, n, C, Y.data_ptr(),
                                       r.data_ptr(), None)
    assert st == mhc.MHC_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert not bool(Y.any()) and not bool(r.any())  # nothing ran


def test_no_alloc_at_its_largest_batch():
    """n=8 at the largest batch whose scratch fits (B = 32,256 on a 152-SM GB300):
    still the results of the workspace call, twice in a row."""
    props = torch.cuda.get_device_properties(0)
    n, C = 8, 8
    B = 32256 if props.multi_processor_count == 152 else 1024
    wl = WORKLOADS["tiny"].with_(B=B, n=n, C=C)
    inp = make_inputs(wl, seed=11, parts=("X", "phi_t"))
    X, phi_t = dev_bf16(inp["X"]), dev_bf16(inp["phi_t"])
    Yw, rw = _with_workspace(X, phi_t, B, n, C)
    for _ in range(2):
        Yn, rn = _no_alloc(X, phi_t, B, n, C)
        torch.cuda.synchronize()
        assert torch.equal(Yn, Yw) and torch.equal(rn, rw)


def test_no_alloc_rejects_host_memory():
    """A page-locked host buffer (reachable by the GPU, so a wrong launch could not
    fault) given as an output is refused before anything is launched."""
    wl = WORKLOADS["tiny"]
    inp = make_inputs(wl, seed=5, parts=("X", "phi_t"))
    X, phi_t = dev_bf16(inp["X"]), dev_bf16(inp["phi_t"])
    N = wl.n * wl.n + 2 * wl.n
    Y_host = torch.zeros(wl.B, N, dtype=torch.float32).pin_memory()
    r = torch.zeros(wl.B, dtype=torch.float32, device="cuda")
    st = mhc._lib.mhc_gemm_rms_noalloc(X.data_ptr(), phi_t.data_ptr(), wl.B, wl.n, wl.C,
                                       Y_host.data_ptr(), r.data_ptr(), None)
    assert st == mhc.MHC_ERR_INVALID
    torch.cuda.synchronize()
    assert not bool(Y_host.any()) and not bool(r.any())


def test_no_alloc_empty_batch_and_bad_shape():
    assert mhc._lib.mhc_gemm_rms_noalloc(None, None, 0, 4, 256, None, None, None) == mhc.MHC_OK
    assert mhc._lib.mhc_gemm_rms_noalloc(None, None, 0, 9, 256, None, None, None) == \
        mhc.MHC_ERR_UNSUPPORTED
