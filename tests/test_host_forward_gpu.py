"""mhc_forward_host: the forward over host-resident activations, chunked through
the device with copies overlapped (include/mhc.h).  Its results must equal
mhc_forward's on the same chunks bit for bit (tokens are independent, page
"mHC 算法分析 & cutile 高效实现" §2.3) and the oracle's within the tolerances.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import (H_TOL, R_REL, assert_abs, assert_bf16_close, assert_rel, assert_Y_close,
                      cuda_ok, dev_bf16, dev_f32, host64, phi_KN)
from synth import WORKLOADS, make_inputs

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]

mhc = pytest.importorskip("gemm_rms_sinkhorn_gb300")

FULL = 1024  # tokens per full chunk of the host pipeline


def chunk_sizes(B):
    """The chunk schedule include/mhc.h states for mhc_forward_host."""
    if B < 2560:
        return [min(256, B - t) for t in range(0, B, 256)]
    mid = B - 1536
    return [256, 512] + [min(FULL, mid - t) for t in range(0, mid, FULL)] + [512, 256]


OUTS = ("Y", "r", "H_pre", "H_post", "H_res", "F_pre", "X_next")


def host_bf16(bits, pin=True):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pin else t.clone()


def run_host(inp, wl, pin=True, in_place=False, scratch=None):
    hX, hF = host_bf16(inp["X"], pin), host_bf16(inp["F_out"], pin)
    out = mhc.alloc_host_outputs(wl.B, wl.n, wl.C, pin=pin)
    if in_place:
        out["X_next"] = hX
    scratch = mhc.host_scratch(wl.B, wl.n, wl.C) if scratch is None else scratch
    mhc.mhc_forward_host(hX, dev_bf16(inp["phi_t"]), hF, wl.alpha_pre, wl.alpha_post,
                         wl.alpha_res, dev_f32(inp["bias"]), wl.iters, wl.B, wl.n, wl.C,
                         out["Y"], out["r"], out["H_pre"], out["H_post"], out["H_res"],
                         out["F_pre"], out["X_next"], scratch)
    torch.cuda.synchronize()
    return out


def device_by_chunks(inp, wl):
    """mhc_forward on each chunk of the batch, on device buffers."""
    parts = {k: [] for k in OUTS}
    phi, bias = dev_bf16(inp["phi_t"]), dev_f32(inp["bias"])
    t0 = 0
    for bc in chunk_sizes(wl.B):
        t1 = t0 + bc
        out = mhc.forward(dev_bf16(inp["X"][t0:t1]), phi, dev_bf16(inp["F_out"][t0:t1]),
                          wl.alpha_pre, wl.alpha_post, wl.alpha_res, bias, wl.iters, wl.n, wl.C)
        torch.cuda.synchronize()
        for k in OUTS:
            parts[k].append(out[k].cpu())
        t0 = t1
    return {k: torch.cat(v) for k, v in parts.items()}


def check_oracle(out, inp, wl):
    ref = oracle.forward(inp["X"], phi_KN(inp["phi_t"]), inp["F_out"], wl.n, wl.C,
                         wl.alpha_pre, wl.alpha_post, wl.alpha_res, inp["bias"], wl.iters)
    g = {k: out[k].double().numpy() for k in OUTS}
    assert_Y_close(g["Y"], ref["Y"], inp["X"], inp["phi_t"])
    assert_rel(g["r"], ref["r"], R_REL, "r")
    for k in ("H_pre", "H_post", "H_res"):
        assert_abs(g[k], ref[k], H_TOL, k)
    assert_bf16_close(g["F_pre"], ref["F_pre"], "F_pre")
    assert_bf16_close(g["X_next"], ref["X_next"].reshape(wl.B, -1), "X_next")


@pytest.mark.parametrize("B,n,C", [(4100, 4, 256), (2100, 8, 64), (5, 3, 24), (2048, 2, 136),
                                   (1024, 4, 7168), (3000, 4, 2048)])
def test_host_forward_equals_device_chunks_and_oracle(B, n, C):
    wl = WORKLOADS["tiny"].with_(B=B, n=n, C=C, bias_std=0.3)
    inp = make_inputs(wl, seed=12)
    out = run_host(inp, wl)
    ref = device_by_chunks(inp, wl)
    for k in OUTS:
        assert torch.equal(out[k].reshape(ref[k].shape), ref[k]), k
    check_oracle(out, inp, wl)


def test_host_forward_in_place_and_pageable():
    wl = WORKLOADS["tiny"].with_(B=4500, C=128)
    inp = make_inputs(wl, seed=13)
    a = run_host(inp, wl)
    b = run_host(inp, wl, pin=False, in_place=True)
    for k in OUTS:
        assert torch.equal(a[k], b[k]), k


def test_host_forward_back_to_back_calls():
    """Two calls enqueued without a sync in between, into the same scratch."""
    wl = WORKLOADS["tiny"].with_(B=4200, C=128)
    inps = [make_inputs(wl, seed=s) for s in (14, 15)]
    scratch = mhc.host_scratch(wl.B, wl.n, wl.C)
    outs = []
    for inp in inps:
        hX, hF = host_bf16(inp["X"]), host_bf16(inp["F_out"])
        out = mhc.alloc_host_outputs(wl.B, wl.n, wl.C)
        mhc.mhc_forward_host(hX, dev_bf16(inp["phi_t"]), hF, wl.alpha_pre, wl.alpha_post,
                             wl.alpha_res, dev_f32(inp["bias"]), wl.iters, wl.B, wl.n, wl.C,
                             out["Y"], out["r"], out["H_pre"], out["H_post"], out["H_res"],
                             out["F_pre"], out["X_next"], scratch)
        outs.append((out, hX, hF))
    torch.cuda.synchronize()
    for (out, _, _), inp in zip(outs, inps):
        check_oracle(out, inp, wl)


def test_host_forward_rejects_device_activations_and_small_scratch():
    wl = WORKLOADS["tiny"]
    inp = make_inputs(wl, seed=16)
    dX, dF = dev_bf16(inp["X"]), dev_bf16(inp["F_out"])
    out = mhc.alloc_host_outputs(wl.B, wl.n, wl.C)
    phi, bias = dev_bf16(inp["phi_t"]), dev_f32(inp["bias"])
    scratch = mhc.host_scratch(wl.B, wl.n, wl.C)
    p = lambda t: t.data_ptr()
    args = [p(dX), p(phi), p(dF), wl.alpha_pre, wl.alpha_post, wl.alpha_res, p(bias), wl.iters,
            wl.B, wl.n, wl.C] + [p(out[k]) for k in OUTS] + [p(scratch), scratch.numel(), None]
    assert mhc._lib.mhc_forward_host(*args) == mhc.MHC_ERR_INVALID  # X on the device
    hX, hF = host_bf16(inp["X"]), host_bf16(inp["F_out"])
    args[0], args[2] = p(hX), p(hF)
    h_phi = host_bf16(inp["phi_t"])
    args[1] = p(h_phi)
    assert mhc._lib.mhc_forward_host(*args) == mhc.MHC_ERR_INVALID  # phi_t on the host
    args[1] = p(phi)
    args[-2] = scratch.numel() - 256
    assert mhc._lib.mhc_forward_host(*args) == mhc.MHC_ERR_WORKSPACE
    args[-2] = scratch.numel()
    assert mhc._lib.mhc_forward_host(*args) == mhc.MHC_OK
    torch.cuda.synchronize()
    check_oracle(out, inp, wl)
    assert mhc.mhc_device_status() == mhc.MHC_OK
