"""Failure detection on the GPU without a fault: a wait inside the GEMM+RMS
kernel is made to run out (one pipeline stage is left unfilled through the
test hook of include/mhc_testing.h, with a 50 ms wait limit).  The kernel must
report MHC_ERR_TIMEOUT through the device status word, return cleanly, and
leave the CUDA context usable for the next call.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import R_REL, assert_rel, assert_Y_close, cuda_ok, dev_bf16, host64, phi_KN
from synth import WORKLOADS, make_inputs

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]

mhc = pytest.importorskip("gemm_rms_sinkhorn_gb300")


def _gemm(X, phi_t, wl, stall_stage=None, limit_ns=50_000_000):
    N = wl.N
    Y = torch.zeros(wl.B, N, dtype=torch.float32, device="cuda")
    r = torch.zeros(wl.B, dtype=torch.float32, device="cuda")
    ws = mhc.workspace(wl.B, wl.n, wl.C)
    stream = torch.cuda.current_stream().cuda_stream
    if stall_stage is None:
        st = mhc._lib.mhc_gemm_rms(X.data_ptr(), phi_t.data_ptr(), wl.B, wl.n, wl.C,
                                   Y.data_ptr(), r.data_ptr(), ws.data_ptr(), ws.numel(), stream)
    else:
        st = mhc._lib.mhc_testing_gemm_rms_stalled(X.data_ptr(), phi_t.data_ptr(), wl.B, wl.n,
                                                   wl.C, Y.data_ptr(), r.data_ptr(),
                                                   ws.data_ptr(), ws.numel(), stall_stage,
                                                   limit_ns, stream)
    assert st == mhc.MHC_OK, mhc.mhc_status_str(st)
    torch.cuda.synchronize()  # a fault would raise here
    return Y, r


@pytest.mark.parametrize("stall_stage", [0, 5])
def test_stalled_wait_reports_timeout_and_context_survives(stall_stage):
    wl = WORKLOADS["decode8"]  # 14 pipeline stages per CTA
    inp = make_inputs(wl, seed=9, parts=("X", "phi_t"))
    X, phi_t = dev_bf16(inp["X"]), dev_bf16(inp["phi_t"])
    assert mhc.mhc_device_status() == mhc.MHC_OK  # clears anything left over
    _gemm(X, phi_t, wl, stall_stage=stall_stage)
    assert mhc.mhc_device_status() == mhc.MHC_ERR_TIMEOUT
    assert mhc.mhc_device_status() == mhc.MHC_OK  # reading cleared it
    # the context is still good: a normal call is correct
    Y, r = _gemm(X, phi_t, wl)
    Yr, rr = oracle.gemm_rms(inp["X"], phi_KN(inp["phi_t"]), wl.n, wl.C)
    assert_Y_close(host64(Y), Yr, inp["X"], inp["phi_t"])
    assert_rel(host64(r), rr, R_REL, "r")
    assert mhc.mhc_device_status() == mhc.MHC_OK


def test_hook_without_stall_is_the_normal_call():
    wl = WORKLOADS["decode32"]
    inp = make_inputs(wl, seed=10, parts=("X", "phi_t"))
    X, phi_t = dev_bf16(inp["X"]), dev_bf16(inp["phi_t"])
    a = _gemm(X, phi_t, wl, stall_stage=-1, limit_ns=4_000_000_000)
    b = _gemm(X, phi_t, wl)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert mhc.mhc_device_status() == mhc.MHC_OK
