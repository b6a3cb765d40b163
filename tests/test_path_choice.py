"""mhc_forward's path choice: the one-launch steps 1-4a kernel for batches of
up to 2048 tokens, the kernel chain above.  The host-side rule runs on CPU;
on the GPU the chosen path is timed against the other one, at sizes where the
measured gap is wide enough for a timing test to be stable (the two paths are
within 2 % of each other at the threshold itself, so that point is not
asserted)."""
import statistics

import pytest

mhc = pytest.importorskip("gemm_rms_sinkhorn_gb300")


@pytest.mark.parametrize("B,n,C,path", [
    (1, 4, 7168, "decode"), (128, 4, 7168, "decode"), (2048, 4, 7168, "decode"),
    (2049, 4, 7168, "chain"), (3072, 4, 7168, "chain"), (4096, 4, 4096, "chain"),
    (16384, 4, 7168, "chain"), (2048, 8, 4096, "decode"), (8192, 8, 4096, "chain"),
    (0, 4, 7168, "chain")])
def test_forward_path_rule(B, n, C, path):
    assert mhc.mhc_testing_forward_path(B, n, C) == path


def test_forward_path_rule_checks_the_shape():
    for B, n, C in ((16, 9, 64), (16, 4, 12), (-1, 4, 64)):
        with pytest.raises(mhc.MhcError):
            mhc.mhc_testing_forward_path(B, n, C)


def _us_per_forward(B, n, C, hook):
    import torch

    from synth import WORKLOADS, make_inputs
    from gpu_util import dev_bf16, dev_f32

    wl = WORKLOADS["tiny"].with_(B=B, n=n, C=C)
    inp = make_inputs(wl, seed=3)
    X = dev_bf16(inp["X"])
    out = mhc.alloc_outputs(B, n, C)
    args = (X, dev_bf16(inp["phi_t"]), dev_bf16(inp["F_out"]), wl.alpha_pre, wl.alpha_post,
            wl.alpha_res, dev_f32(inp["bias"]), wl.iters, B, n, C, out["Y"], out["r"],
            out["H_pre"], out["H_post"], out["H_res"], out["F_pre"], out["X_next"], out["ws"])
    fn = getattr(mhc, hook)
    for _ in range(5):
        fn(*args)
    times = []
    for _ in range(7):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(10):
            fn(*args)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 100.0)  # µs per forward
    return statistics.median(times)


@pytest.mark.gpu
@pytest.mark.parametrize("B,n,C,margin", [(128, 4, 7168, 1.2), (1024, 4, 7168, 1.05),
                                          (512, 8, 4096, 1.5)])
def test_small_batches_take_the_faster_path(B, n, C, margin):
    """Below the threshold the one-launch path is chosen and is faster than the
    chain by at least `margin` (stream launches, measured: B=128, n=4, C=7168:
    24-29 against 39 µs; B=1024: 49-50 against 56 µs; B=512, n=8, C=4096: 43
    against 119 µs)."""
    assert mhc.mhc_testing_forward_path(B, n, C) == "decode"
    decode = _us_per_forward(B, n, C, "mhc_testing_forward_decode")
    chain = _us_per_forward(B, n, C, "mhc_testing_forward_chain")
    assert decode * margin < chain, (decode, chain)


@pytest.mark.gpu
@pytest.mark.parametrize("B,n,C", [(3072, 4, 7168), (4096, 4, 7168), (3072, 8, 4096)])
def test_above_the_threshold_the_chain_is_not_slower(B, n, C):
    """Above 2048 tokens the chain is chosen; measured (stream launches) 130
    against 136 µs at B=3072, n=4, C=7168, 169 against 179 µs at 4096, and 161
    against 171 µs at B=3072, n=8, C=4096: it must not be more than 5 % slower."""
    assert mhc.mhc_testing_forward_path(B, n, C) == "chain"
    decode = _us_per_forward(B, n, C, "mhc_testing_forward_decode")
    chain = _us_per_forward(B, n, C, "mhc_testing_forward_chain")
    assert chain < 1.05 * decode, (chain, decode)
