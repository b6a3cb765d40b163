"""Failure detection on the GPU without a fault: a wait inside a kernel is
made to run out through the test hooks of include/mhc_testing.h, with a 50 ms
wait limit: one pipeline stage of the GEMM+RMS kernel left unfilled, or the
grid barrier of the small-batch forward kernel waiting for one CTA more than
the grid has.  The kernel must report MHC_ERR_TIMEOUT through the device
status word, return cleanly, and leave the CUDA context usable for the next
call.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import (H_TOL, R_REL, assert_abs, assert_bf16_close, assert_rel, assert_Y_close,
                      cuda_ok, dev_bf16, dev_f32, host64, phi_KN)
from synth import WORKLOADS, Workload, make_inputs

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


def _forward(inp, wl, stalled=False):
    X = dev_bf16(inp["X"])
    out = {k: v.zero_() for k, v in mhc.alloc_outputs(wl.B, wl.n, wl.C).items()}
    args = (X, dev_bf16(inp["phi_t"]), dev_bf16(inp["F_out"]), wl.alpha_pre, wl.alpha_post,
            wl.alpha_res, dev_f32(inp["bias"]), wl.iters, wl.B, wl.n, wl.C, out["Y"], out["r"],
            out["H_pre"], out["H_post"], out["H_res"], out["F_pre"], out["X_next"], out["ws"])
    if stalled:
        mhc.mhc_testing_forward_decode_stalled(*args, 50_000_000)
    else:
        mhc.mhc_testing_forward_decode(*args)
    torch.cuda.synchronize()  # a fault would raise here
    return out


def test_stalled_grid_barrier_reports_timeout_and_context_survives():
    wl = WORKLOADS["decode32"]
    inp = make_inputs(wl, seed=11)
    assert mhc.mhc_device_status() == mhc.MHC_OK
    out = _forward(inp, wl, stalled=True)
    assert mhc.mhc_device_status() == mhc.MHC_ERR_TIMEOUT
    # no CTA passed the barrier, so nothing of steps 1-4a was written, nor
    # X_next, which the same kernel forms at this batch size
    for k in ("Y", "r", "H_pre", "H_post", "H_res", "F_pre", "X_next"):
        assert not bool(out[k].any()), k
    assert mhc.mhc_device_status() == mhc.MHC_OK
    out = _forward(inp, wl)
    ref = oracle.forward(inp["X"], phi_KN(inp["phi_t"]), inp["F_out"], wl.n, wl.C, wl.alpha_pre,
                         wl.alpha_post, wl.alpha_res, inp["bias"], wl.iters)
    assert_Y_close(host64(out["Y"]), ref["Y"], inp["X"], inp["phi_t"])
    assert_rel(host64(out["r"]), ref["r"], R_REL, "r")
    assert_abs(host64(out["H_res"]), ref["H_res"], H_TOL, "H_res")
    assert_bf16_close(host64(out["F_pre"]), ref["F_pre"], "F_pre")
    assert_bf16_close(host64(out["X_next"]), ref["X_next"], "X_next")
    assert mhc.mhc_device_status() == mhc.MHC_OK


def _forward_ws(inp, wl, out, ws, stalled=False, stream=None):
    args = (inp["Xd"], inp["phid"], inp["Fd"], wl.alpha_pre, wl.alpha_post, wl.alpha_res,
            inp["biasd"], wl.iters, wl.B, wl.n, wl.C, out["Y"], out["r"], out["H_pre"],
            out["H_post"], out["H_res"], out["F_pre"], out["X_next"], ws)
    if stalled:
        mhc.mhc_testing_forward_decode_stalled(*args, 50_000_000, stream=stream)
    else:
        mhc.mhc_testing_forward_decode(*args, stream=stream)


def _device_inputs(wl, seed):
    inp = make_inputs(wl, seed=seed)
    inp.update(Xd=dev_bf16(inp["X"]), phid=dev_bf16(inp["phi_t"]), Fd=dev_bf16(inp["F_out"]),
               biasd=dev_f32(inp["bias"]))
    return inp


@pytest.mark.parametrize("wl_name", ["decode8", "decode128"])
def test_grid_barrier_words_clear_themselves(wl_name):
    """The small-batch kernel's grid barrier needs no zeroed workspace: its
    words carry the launch's epoch, start from whatever the workspace holds
    and are 0 again when the kernel ends, after a completed barrier and after
    one whose wait ran out."""
    wl = WORKLOADS[wl_name]
    inp = _device_inputs(wl, seed=12)
    ref_out = mhc.alloc_outputs(wl.B, wl.n, wl.C)
    _forward_ws(inp, wl, ref_out, ref_out["ws"])
    torch.cuda.synchronize()
    assert mhc.mhc_device_status() == mhc.MHC_OK
    out = {k: torch.empty_like(v) for k, v in ref_out.items()}
    ws = out["ws"]
    for fill in (0xA5, 0x00, 0xFF):
        ws.fill_(fill)
        _forward_ws(inp, wl, out, ws)
        torch.cuda.synchronize()
        assert mhc.mhc_device_status() == mhc.MHC_OK
        assert not bool(ws[:16].any()), "barrier words left set"
        for k in ("Y", "r", "H_pre", "H_post", "H_res", "F_pre", "X_next"):
            assert torch.equal(out[k], ref_out[k]), k
    _forward_ws(inp, wl, out, ws, stalled=True)
    torch.cuda.synchronize()
    assert mhc.mhc_device_status() == mhc.MHC_ERR_TIMEOUT
    assert not bool(ws[:16].any()), "barrier words left set after a timeout"
    _forward_ws(inp, wl, out, ws)
    torch.cuda.synchronize()
    assert mhc.mhc_device_status() == mhc.MHC_OK
    for k in ("Y", "r", "H_pre", "H_post", "H_res", "F_pre", "X_next"):
        assert torch.equal(out[k], ref_out[k]), k


@pytest.mark.parametrize("B", [32, 512])
def test_grid_barrier_in_a_replayed_graph(B):
    """A CUDA graph fixes the launch's epoch, so every replay meets words that
    the previous replay cleared; the replays give the eager call's bits.  At
    B = 512 the X_next kernel runs between two launches of the small-batch
    kernel."""
    wl = Workload(f"decode{B}", B=B, n=4, C=7168)
    inp = _device_inputs(wl, seed=13)
    ref_out = mhc.alloc_outputs(wl.B, wl.n, wl.C)
    _forward_ws(inp, wl, ref_out, ref_out["ws"])
    torch.cuda.synchronize()
    out = {k: torch.zeros_like(v) for k, v in ref_out.items()}
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for _ in range(3):
                _forward_ws(inp, wl, out, out["ws"], stream=side)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(4):
        for k in ("Y", "H_res", "F_pre", "X_next"):
            out[k].zero_()
        g.replay()
        torch.cuda.synchronize()
        assert mhc.mhc_device_status() == mhc.MHC_OK
        assert not bool(out["ws"][:16].any())
        for k in ("Y", "r", "H_pre", "H_post", "H_res", "F_pre", "X_next"):
            assert torch.equal(out[k], ref_out[k]), k
