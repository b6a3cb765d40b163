"""Out-of-bounds writes and foreign pointers, on the GPU, through the C ABI.

Guard bytes: every buffer a call receives (inputs, outputs and the workspace)
sits inside a larger allocation with GUARD bytes of a seeded byte pattern on
each side.  After the call the guards must be unchanged, and so must every
input.  A kernel that wrote past the end of an output (a ragged last token
tile, a split-K park slot, the grid-barrier word, the chunk slots of the
host-buffer forward) would change them.  Shapes cover one token, odd token
counts around the 128-token tiles, and K that is not a multiple of the 64-wide
K blocks.

Pointer kinds: page-locked host memory handed to a device entry point (or
device memory handed to mhc_forward_host where host memory is expected) must
be refused with MHC_ERR_INVALID before anything is launched.  Page-locked
memory is reachable by the GPU, so even a regression could not fault.
"""

import pytest
import torch

from gpu_util import cuda_ok

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA device")]

mhc = pytest.importorskip("gemm_rms_sinkhorn_gb300")
L = mhc._lib

GUARD = 4096
BS = [1, 3, 65, 129, 4097]
NS = list(range(1, 9))


def _pattern(nbytes, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g)


class Arena:
    """Buffers with guard bytes on both sides, device or page-locked host."""

    def __init__(self, seed):
        self.bufs = {}
        self.seed = seed

    def add(self, name, nbytes, role, host=False, fill="random"):
        size = (max(nbytes, 1) + 15) // 16 * 16
        total = GUARD + size + GUARD
        pat = _pattern(total, self.seed * 131 + len(self.bufs))
        if fill == "zero":
            pat[GUARD:GUARD + size] = 0
        elif fill == "bf16":  # finite bf16 values in [-2, 2): keeps the arithmetic in range
            v = (torch.rand(size // 2, generator=torch.Generator().manual_seed(len(self.bufs)))
                 * 4 - 2).to(torch.bfloat16)
            pat[GUARD:GUARD + size] = v.view(torch.uint8)
        elif fill == "f32":
            v = torch.rand(size // 4, generator=torch.Generator().manual_seed(len(self.bufs))) + 0.5
            pat[GUARD:GUARD + size] = v.view(torch.uint8)
        elif fill == "e4m3":  # finite e4m3 codes: clear the 0x7F/0xFF NaN pattern
            pat[GUARD:GUARD + size] &= 0x77
        t = pat.pin_memory() if host else pat.cuda()
        self.bufs[name] = dict(t=t, ref=pat, nbytes=nbytes, size=size, role=role)
        return t.data_ptr() + GUARD

    def ptr(self, name):
        return self.bufs[name]["t"].data_ptr() + GUARD

    def check(self, where, skip_inputs=()):
        torch.cuda.synchronize()
        for name, b in self.bufs.items():
            got = b["t"].cpu()
            ref = b["ref"]
            lo, hi = GUARD, GUARD + b["nbytes"]
            assert torch.equal(got[:lo], ref[:lo]), "%s: guard before %s written" % (where, name)
            assert torch.equal(got[hi:], ref[hi:]), "%s: guard after %s written" % (where, name)
            if b["role"] == "in" and name not in skip_inputs:
                assert torch.equal(got[lo:hi], ref[lo:hi]), "%s: input %s changed" % (where, name)


def _sizes(B, n, C, e4m3=False):
    N, K = n * n + 2 * n, n * C
    act = 1 if e4m3 else 2
    return dict(X=B * K * act, phi=N * K * act, Fo=B * C * act, bias=N * 4, Y=B * N * 4, r=B * 4,
                hp=B * n * 4, hq=B * n * 4, hr=B * n * n * 4, Fp=B * C * act,
                Xn=B * K * act)


def _forward_arena(B, n, C, seed, e4m3=False, f32w=False, host=False):
    s = _sizes(B, n, C, e4m3)
    a = Arena(seed)
    act = "e4m3" if e4m3 else "bf16"
    a.add("X", s["X"], "in", host=host, fill=act)
    phi = s["phi"] * (2 if f32w else 1)
    a.add("phi", phi, "in", fill=act)
    a.add("Fo", s["Fo"] * (2 if f32w else 1), "in", host=host, fill="f32" if f32w else act)
    a.add("bias", s["bias"], "in", fill="f32")
    for k in ("Y", "r", "hp", "hq", "hr", "Fp", "Xn"):
        a.add(k, s[k], "out", host=host)
    if host:
        ws = L.mhc_forward_host_scratch_bytes(B, n, C)
    else:
        ws = L.mhc_workspace_bytes(B, n, C)
    a.add("ws", ws, "ws")
    return a, ws


def _fwd_args(a, B, n, C, ws):
    p = a.ptr
    return (p("X"), p("phi"), p("Fo"), 0.01, 0.01, 0.01, p("bias"), 20, B, n, C, p("Y"), p("r"),
            p("hp"), p("hq"), p("hr"), p("Fp"), p("Xn"), p("ws"), ws, None)


FORWARDS = ["mhc_forward", "mhc_testing_forward_chain", "mhc_testing_forward_decode",
            "mhc_testing_forward_fused"]


@pytest.mark.parametrize("C", [8, 264])
@pytest.mark.parametrize("B", BS)
@pytest.mark.parametrize("entry", FORWARDS)
def test_forward_paths_write_only_their_outputs(entry, B, C):
    for n in NS:
        a, ws = _forward_arena(B, n, C, seed=B * 10 + n)
        st = getattr(L, entry)(*_fwd_args(a, B, n, C, ws))
        assert st in (mhc.MHC_OK, mhc.MHC_ERR_UNSUPPORTED), (entry, B, n, C, st)
        if entry == "mhc_forward":
            assert st == mhc.MHC_OK
        a.check("%s B=%d n=%d C=%d" % (entry, B, n, C))
    assert mhc.mhc_device_status() == mhc.MHC_OK


# shapes the one-kernel steps 1-4a path accepts (two or more token tiles), ragged
@pytest.mark.parametrize("B,n,C", [(1000, 4, 7168), (4097, 3, 2048), (600, 8, 2048),
                                   (4097, 2, 1024), (257, 1, 8192), (300, 5, 2048)])
def test_fused_path_writes_only_its_outputs(B, n, C):
    a, ws = _forward_arena(B, n, C, seed=7)
    assert L.mhc_testing_forward_fused(*_fwd_args(a, B, n, C, ws)) == mhc.MHC_OK
    a.check("fused B=%d n=%d C=%d" % (B, n, C))


@pytest.mark.parametrize("C", [16, 272])
@pytest.mark.parametrize("B", BS)
def test_e4m3_forward_writes_only_its_outputs(B, C):
    for n in NS:
        a, ws = _forward_arena(B, n, C, seed=B + n, e4m3=True)
        assert L.mhc_forward_e4m3(*_fwd_args(a, B, n, C, ws)) == mhc.MHC_OK
        a.check("e4m3 B=%d n=%d C=%d" % (B, n, C))


@pytest.mark.parametrize("C", [8, 264])
@pytest.mark.parametrize("B", BS)
def test_f32w_forward_writes_only_its_outputs(B, C):
    for n in NS:
        a, ws = _forward_arena(B, n, C, seed=B + 3 * n, f32w=True)
        assert L.mhc_forward_f32w(*_fwd_args(a, B, n, C, ws)) == mhc.MHC_OK
        a.check("f32w B=%d n=%d C=%d" % (B, n, C))


@pytest.mark.parametrize("B", [1, 3, 129, 4097])
def test_host_forward_writes_only_its_outputs(B):
    for n, C in [(1, 8), (4, 264), (8, 264), (3, 8)]:
        a, ws = _forward_arena(B, n, C, seed=B + n, host=True)
        assert L.mhc_forward_host(*_fwd_args(a, B, n, C, ws)) == mhc.MHC_OK
        a.check("host B=%d n=%d C=%d" % (B, n, C))


@pytest.mark.parametrize("C", [8, 264])
@pytest.mark.parametrize("B", BS)
def test_single_calls_write_only_their_outputs(B, C):
    """mhc_gemm_rms (+ _noalloc, _coeffs, _split), mhc_coeffs and the apply calls (bf16,
    fp32 F_out, e4m3) one by one."""
    for n in NS:
        N, K = n * n + 2 * n, n * C
        s = _sizes(B, n, C)
        a = Arena(B * 7 + n)
        X = a.add("X", s["X"], "in", fill="bf16")
        phi = a.add("phi", s["phi"], "in", fill="bf16")
        phi2 = a.add("phi2", 2 * s["phi"], "in", fill="bf16")
        phi32 = a.add("phi32", 2 * s["phi"], "in", fill="f32")
        bias = a.add("bias", s["bias"], "in", fill="f32")
        Fo = a.add("Fo", s["Fo"], "in", fill="bf16")
        Fo32 = a.add("Fo32", 2 * s["Fo"], "in", fill="f32")
        Yi = a.add("Yi", s["Y"], "in", fill="f32")
        ri = a.add("ri", s["r"], "in", fill="f32")
        hpi = a.add("hpi", s["hp"], "in", fill="f32")
        hqi = a.add("hqi", s["hq"], "in", fill="f32")
        hri = a.add("hri", s["hr"], "in", fill="f32")
        X8 = a.add("X8", B * K, "in", fill="e4m3")
        Fo8 = a.add("Fo8", B * C, "in", fill="e4m3")
        outs = {}
        for k, nb in [("Y", s["Y"]), ("r", s["r"]), ("hp", s["hp"]), ("hq", s["hq"]),
                      ("hr", s["hr"]), ("Fp", s["Fp"]), ("Xn", s["Xn"]), ("split", 2 * s["phi"]),
                      ("Y2", s["Y"]), ("r2", s["r"]), ("Y3", s["Y"]), ("r3", s["r"]),
                      ("Xn2", s["Xn"]), ("Fp8", B * C), ("Xn8", B * K), ("Y4", s["Y"]),
                      ("r4", s["r"]), ("Y5", s["Y"]), ("r5", s["r"]), ("hp5", s["hp"]),
                      ("hq5", s["hq"]), ("hr5", s["hr"])]:
            outs[k] = a.add(k, nb, "out")
        ws_n = L.mhc_workspace_bytes(B, n, C)
        ws = a.add("ws", ws_n, "ws")
        calls = [
            ("gemm_rms", L.mhc_gemm_rms(X, phi, B, n, C, outs["Y"], outs["r"], ws, ws_n, None)),
            ("noalloc", L.mhc_gemm_rms_noalloc(X, phi, B, n, C, outs["Y2"], outs["r2"], None)),
            ("split_phi", L.mhc_split_phi(phi32, n, C, outs["split"], None)),
            ("gemm_rms_split", L.mhc_gemm_rms_split(X, phi2, B, n, C, outs["Y3"], outs["r3"], ws,
                                                     ws_n, None)),
            ("gemm_rms_e4m3", L.mhc_gemm_rms_e4m3(X8, phi, B, n, C, outs["Y4"], outs["r4"], ws,
                                                   ws_n, None) if C % 16 == 0 else mhc.MHC_OK),
            ("coeffs", L.mhc_coeffs(Yi, ri, 0.01, 0.01, 0.01, bias, 20, B, n, outs["hp"],
                                    outs["hq"], outs["hr"], None)),
            ("gemm_rms_coeffs", L.mhc_gemm_rms_coeffs(X, phi, 0.01, 0.01, 0.01, bias, 20, B, n, C,
                                                      outs["Y5"], outs["r5"], outs["hp5"],
                                                      outs["hq5"], outs["hr5"], ws, ws_n, None)),
            ("pre_apply", L.mhc_pre_apply(X, hpi, B, n, C, outs["Fp"], None)),
            ("post_res_apply", L.mhc_post_res_apply(X, Fo, hri, hqi, B, n, C, outs["Xn"], None)),
            ("post_res_apply_f32", L.mhc_post_res_apply_f32(X, Fo32, hri, hqi, B, n, C,
                                                            outs["Xn2"], None)),
        ]
        if C % 16 == 0:
            calls += [("pre_apply_e4m3", L.mhc_pre_apply_e4m3(X8, hpi, B, n, C, outs["Fp8"], None)),
                      ("post_res_apply_e4m3", L.mhc_post_res_apply_e4m3(X8, Fo8, hri, hqi, B, n, C,
                                                                        outs["Xn8"], None))]
        for name, st in calls:
            assert st == mhc.MHC_OK, (name, B, n, C, mhc.mhc_status_str(st))
        a.check("single calls B=%d n=%d C=%d" % (B, n, C))


@pytest.mark.parametrize("M,K,N", [(1, 8, 8), (3, 264, 72), (65, 8, 264), (129, 264, 8),
                                   (4097, 264, 264), (300, 4096, 512), (16384, 2048, 40)])
def test_rmsnorm_gemm_writes_only_its_output(M, K, N):
    a = Arena(M + K + N)
    A = a.add("A", M * K * 2, "in", fill="bf16")
    Bt = a.add("Bt", N * K * 2, "in", fill="bf16")
    C = a.add("C", M * N * 2, "out")
    ws_n = L.mhc_rmsnorm_gemm_workspace_bytes(M, K, N)
    ws = a.add("ws", ws_n, "ws")
    assert L.mhc_rmsnorm_gemm(A, Bt, M, K, N, 1e-5, C, ws, ws_n, None) == mhc.MHC_OK
    a.check("rmsnorm_gemm M=%d K=%d N=%d" % (M, K, N))


# ------------------------------------------------------------ pointer kinds


def _host_swap_cases():
    """(entry, argument index that gets a page-locked host buffer) for the device calls."""
    return [("mhc_forward", 0), ("mhc_forward", 11), ("mhc_forward", 17), ("mhc_forward", 18),
            ("mhc_testing_forward_decode", 16), ("mhc_forward_f32w", 2),
            ("mhc_forward_e4m3", 12)]


@pytest.mark.parametrize("entry,arg", _host_swap_cases())
def test_device_calls_refuse_host_memory(entry, arg):
    B, n, C = 65, 4, 272
    a, ws = _forward_arena(B, n, C, seed=3, e4m3=entry.endswith("e4m3"),
                           f32w=entry.endswith("f32w"))
    args = list(_fwd_args(a, B, n, C, ws))
    host = torch.zeros(64 << 20, dtype=torch.uint8).pin_memory()
    args[arg] = host.data_ptr()
    assert getattr(L, entry)(*args) == mhc.MHC_ERR_INVALID
    a.check("%s with host arg %d" % (entry, arg))
    assert not bool(host.any())


def test_single_device_calls_refuse_host_memory():
    B, n, C = 65, 4, 264
    N, K = n * n + 2 * n, n * C
    dev = lambda nb: torch.zeros(nb, dtype=torch.uint8, device="cuda")
    hostb = lambda nb: torch.zeros(nb, dtype=torch.uint8).pin_memory()
    X, phi, Y, r = dev(B * K * 2), dev(N * K * 2), dev(B * N * 4), dev(B * 4)
    ws = dev(max(16, L.mhc_workspace_bytes(B, n, C)))
    Xh, Yh = hostb(B * K * 2), hostb(B * N * 4)
    wsb = ws.numel()
    assert L.mhc_gemm_rms(Xh.data_ptr(), phi.data_ptr(), B, n, C, Y.data_ptr(), r.data_ptr(),
                          ws.data_ptr(), wsb, None) == mhc.MHC_ERR_INVALID
    assert L.mhc_gemm_rms(X.data_ptr(), phi.data_ptr(), B, n, C, Yh.data_ptr(), r.data_ptr(),
                          ws.data_ptr(), wsb, None) == mhc.MHC_ERR_INVALID
    wsh = hostb(wsb)
    assert L.mhc_gemm_rms(X.data_ptr(), phi.data_ptr(), B, n, C, Y.data_ptr(), r.data_ptr(),
                          wsh.data_ptr(), wsb, None) == mhc.MHC_ERR_INVALID
    Fp_h = hostb(B * C * 2)
    Hp = dev(B * n * 4)
    assert L.mhc_pre_apply(X.data_ptr(), Hp.data_ptr(), B, n, C, Fp_h.data_ptr(),
                           None) == mhc.MHC_ERR_INVALID
    Ch = hostb(B * 72 * 2)
    assert L.mhc_rmsnorm_gemm(X.data_ptr(), phi.data_ptr(), B, 264, 72, 1e-5, Ch.data_ptr(),
                              None, 0, None) == mhc.MHC_ERR_INVALID
    torch.cuda.synchronize()
    for t in (Y, r, Yh, wsh, Fp_h, Ch):
        assert not bool(t.any())


def test_host_forward_refuses_device_activations():
    B, n, C = 65, 4, 264
    a, ws = _forward_arena(B, n, C, seed=5, host=True)
    args = list(_fwd_args(a, B, n, C, ws))
    Xd = torch.zeros(B * n * C * 2, dtype=torch.uint8, device="cuda")
    args[0] = Xd.data_ptr()
    assert L.mhc_forward_host(*args) == mhc.MHC_ERR_INVALID
    a.check("host forward with a device X")
