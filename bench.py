#!/usr/bin/env python3
"""Benchmark of the mHC forward hot path on GB300 (one JSON line on rank 0).

A step is one ``mhc_forward`` (GEMM+RMS, coefficients + Sinkhorn, pre-apply,
post/res-apply) over one batch of the prefill workload B=16384, n=4, C=7168
(X 940 MB bf16), inputs resident in HBM.  X is far larger than L2 (129 MB),
so no L2 flush is needed between steps.

Reported:
  value        tokens/s over all ranks (weak scaling: every rank runs its own batch)
  e2e          the same metric through the public C-ABI call over host buffers
               (mhc_forward_host, pinned memory): H2D of the step's inputs X and
               F_out, the forward, D2H of every output, all timed (the call
               overlaps them chunk by chunk; the weights stay on the device)
  roofline     the dominant kernel's algorithmic bytes / its CUDA-event time,
               against the measured HBM copy bandwidth (MEASURED_PEAKS.json)
  cpu_baseline the fp64 oracle split by token range over every host core, with its
               one-core rate beside it, on a bounded token sample
  clocks       nvidia-smi samples taken while the timed steps run

``--impl reference`` times the fp64 oracle instead (every host core, no GPU).
Under torchrun (N > 1) each rank drives its own GPU; rank 0 prints.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "mHC fwd tokens/s & achieved HBM GB/s vs ~8 TB/s (B=16384,n=4,C=7168)"
WORKLOAD = "prefill"
FALLBACK_HBM_GBS = 6800.0
# The kernels of a prefill forward step (the chain): gemm_rms is the GEMM whose
# finalize also forms the coefficients (steps 1-3, mhc_gemm_rms_coeffs).
KERNELS = ("gemm_rms", "pre_apply", "post_res_apply")
# kernel -> source file whose contents the stored DRAM counters were taken from
KERNEL_SOURCES = {"gemm_rms": "gemm_rms.cu", "pre_apply": "apply.cu",
                  "post_res_apply": "apply.cu"}
# Kernels one prefill forward step launches (the chain, far above the small-batch
# threshold of 2048 tokens): zero_tickets_kernel (the split-K tile counters of the
# caller's workspace), gemm_rms_kernel, pre_apply_kernel and post_res_apply_kernel.
LAUNCHES_PER_STEP = 4


def algorithmic_bytes(B: int, n: int, C: int, precision: str = "bf16") -> dict:
    """Compulsory HBM bytes per launch of each kernel (read once, write once).
    precision "f32w": the weight as split bf16 pairs (2·N rows) and F_out fp32."""
    K, N = n * C, n * n + 2 * n
    X, Fc = 2 * B * K, 2 * B * C
    H = 4 * B * (2 * n + n * n)
    wrows = 2 * N if precision == "f32w" else N
    f_in = 4 * B * C if precision == "f32w" else Fc
    wbytes = 2 * wrows * K
    if precision == "e4m3":  # one byte per activation and weight value
        X, Fc, f_in, wbytes = B * K, B * C, B * C, N * K
    return {
        "gemm_rms": X + wbytes + 4 * B * N + 4 * B,
        "coeffs": 4 * B * N + 4 * B + 4 * N + H,
        "pre_apply": X + 4 * B * n + Fc,
        "post_res_apply": X + f_in + 4 * B * n * n + 4 * B * n + X,
    }


def kernel_bytes(B: int, n: int, C: int, precision: str = "bf16") -> dict:
    """Compulsory HBM bytes per launch of each kernel of KERNELS: the steps of
    algorithmic_bytes, steps 1-3 in one kernel (Y and r written, not read back)."""
    a = algorithmic_bytes(B, n, C, precision)
    N = n * n + 2 * n
    return {"gemm_rms": a["gemm_rms"] + a["coeffs"] - (4 * B * N + 4 * B),
            "pre_apply": a["pre_apply"], "post_res_apply": a["post_res_apply"]}


def measured_peaks() -> tuple:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "MEASURED_PEAKS.json hbm_gbs (of measured)"
    except Exception:
        return FALLBACK_HBM_GBS, "profiling-recipe fallback 6.8 TB/s (of fallback)"


def source_digest(kernel: str) -> str:
    """First 16 hex digits of the SHA-256 over the kernel's .cu file followed by
    every header under csrc/ (sorted), so a change to shared device code also
    marks a stored capture as stale."""
    csrc = os.path.join(ROOT, "gemm_rms_sinkhorn_gb300", "csrc")
    h = hashlib.sha256()
    names = [KERNEL_SOURCES[kernel]] + sorted(f for f in os.listdir(csrc)
                                              if f.endswith((".cuh", ".h")))
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def stored_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu capture, or None if stale/absent."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d[kernel]
        if ent.get("source_sha256_16") != source_digest(kernel):
            return None
        return int(ent["bytes_per_launch"])
    except Exception:
        return None


# ------------------------------------------------------------------ clocks


class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) with host arrival times."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        win = [p for (t, p) in self.samples if t0 <= t <= t1]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[0]) for p in win if num(p[0]) is not None]
        mx = [num(p[1]) for p in win if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4) if p[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "power_w_max": max((num(p[2]) or 0.0) for p in win), "samples": len(win)}


# ------------------------------------------------------------ CPU oracle


def cpu_oracle_rate(wl, inp, budget_s: float, chunk: int = 128):
    """Tokens/s of the fp64 oracle forward on one core: the first tokens of the
    workload, in chunks of `chunk` tokens until `budget_s` seconds of oracle time."""
    import oracle

    phi = np.ascontiguousarray(inp["phi_t"].T)
    done, elapsed = 0, 0.0
    B = inp["X"].shape[0]
    while elapsed < budget_s and done < B:
        rows = min(chunk, B - done)
        X, F = inp["X"][done:done + rows], inp["F_out"][done:done + rows]
        t = time.perf_counter()
        oracle.forward(X, phi, F, wl.n, wl.C, wl.alpha_pre, wl.alpha_post, wl.alpha_res,
                       inp["bias"], wl.iters)
        elapsed += time.perf_counter() - t
        done += rows
    return done / elapsed, done, elapsed


class OracleOnAllCores:
    """The same single-threaded fp64 oracle forward, split by token range over a
    pool of host threads (tokens are independent; the oracle's C call releases
    the GIL).  Outputs land in per-range buffers and are discarded."""

    def __init__(self, wl, inp, workers: int = 0, chunk: int = 32):
        import concurrent.futures

        import oracle

        self.oracle = oracle
        self.wl, self.inp, self.chunk = wl, inp, chunk
        self.phi = np.ascontiguousarray(inp["phi_t"].T)
        self.workers = workers or os.cpu_count() or 1
        self.pool = concurrent.futures.ThreadPoolExecutor(self.workers)

    def _part(self, lo, hi):
        wl, inp = self.wl, self.inp
        self.oracle.forward(inp["X"][lo:hi], self.phi, inp["F_out"][lo:hi], wl.n, wl.C,
                            wl.alpha_pre, wl.alpha_post, wl.alpha_res, inp["bias"], wl.iters)

    def run(self, lo: int, hi: int) -> None:
        futs = [self.pool.submit(self._part, a, min(a + self.chunk, hi))
                for a in range(lo, hi, self.chunk)]
        for f in futs:
            f.result()

    def rate(self, tokens: int):
        """Tokens/s over the first `tokens` tokens (wall clock, all workers)."""
        t = time.perf_counter()
        self.run(0, tokens)
        return tokens / (time.perf_counter() - t), time.perf_counter() - t

    def close(self):
        self.pool.shutdown()


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def run_reference(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    # each step: the oracle forward over a bounded sample of the workload's tokens,
    # split by token range over every host core
    cores = os.cpu_count() or 1
    tokens_per_step = args.ref_tokens or 32 * cores
    import synth

    inp = synth.make_inputs(wl, 0, rows=tokens_per_step)
    pool = OracleOnAllCores(wl, inp, cores)

    for _ in range(args.warmup):
        pool.run(0, tokens_per_step)
    t = time.perf_counter()
    for _ in range(args.steps):
        pool.run(0, tokens_per_step)
    el = time.perf_counter() - t
    pool.close()
    value = tokens_per_step * args.steps / el
    sample = ("first %d tokens of %s per step (fp64 oracle, split by token range over %d "
              "host threads)" % (tokens_per_step, wl.name, cores))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1000.0 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded counter-based generator)",
        "config": workload_config(wl, 1),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample, "cpu": cpu_model()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(wl, world):
    return {"workload": "mHC forward prefill B=%d n=%d C=%d iters=%d" % (wl.B, wl.n, wl.C,
                                                                         wl.iters),
            "B_per_gpu": wl.B, "n": wl.n, "C": wl.C, "K": wl.K, "N": wl.N, "iters": wl.iters,
            "global_batch_tokens": wl.B * world, "parallelism": "replicas%d" % world,
            "l2": "no flush: inputs larger than L2 (X %.0f MB > 129 MB)" % (2 * wl.B * wl.K / 1e6)}


# ------------------------------------------------------- rank combination


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The slowest rank's time: every rank gets the maximum of `x`."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def tokens_per_second(tokens_per_rank: int, world: int, steps: int, ms_total: float) -> float:
    """Whole-job throughput: the tokens every rank processed over the slowest rank's time."""
    return tokens_per_rank * world * steps / (ms_total / 1e3)


# ------------------------------------------------------------------ GPU arm


def forward_latency(mhc, step, stream, barrier, steps, warmup) -> dict:
    """Microseconds per mhc_forward: back-to-back stream launches (includes the
    host's call overhead when it exceeds the GPU time) and replays of a CUDA
    graph holding `steps` forwards (GPU time only)."""
    import torch

    for _ in range(max(warmup, 3)):
        step()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    barrier()
    us_stream = 1e3 * e0.elapsed_time(e1) / steps
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for _ in range(steps):
                step_on = torch.cuda.current_stream()
                step(step_on)
    stream.wait_stream(side)
    for _ in range(2):
        g.replay()
    barrier()
    reps = 5
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    barrier()
    us_graph = 1e3 * e0.elapsed_time(e1) / (reps * steps)
    return {"us_per_forward_stream": us_stream, "us_per_forward_graph": us_graph,
            "forwards_timed": steps}


def per_kernel_times(mhc, stream, barrier, steps, wl, X, phi_t, F_out, bias, out) -> dict:
    """Mean CUDA-event time (ms) of each kernel over `steps` passes of the three
    entry points of the chain, events recorded between launches on the launching stream."""
    runs = per_kernel_runs(mhc, stream, barrier, steps, wl, X, phi_t, F_out, bias, out)
    return {k: statistics.mean(v) for k, v in runs.items()}


def per_kernel_runs(mhc, stream, barrier, steps, wl, X, phi_t, F_out, bias, out) -> dict:
    """CUDA-event time (ms) of each kernel in each of `steps` passes of the three
    entry points of the chain (a list per kernel)."""
    import torch

    B, n, C = wl.B, wl.n, wl.C
    nk = len(KERNELS)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(steps)]
    barrier()
    for s in range(steps):
        e = evs[s]
        e[0].record(stream)
        mhc.mhc_gemm_rms_coeffs(X, phi_t, wl.alpha_pre, wl.alpha_post, wl.alpha_res, bias,
                                wl.iters, B, n, C, out["Y"], out["r"], out["H_pre"],
                                out["H_post"], out["H_res"], out["ws"], stream)
        e[1].record(stream)
        mhc.mhc_pre_apply(X, out["H_pre"], B, n, C, out["F_pre"], stream)
        e[2].record(stream)
        mhc.mhc_post_res_apply(X, F_out, out["H_res"], out["H_post"], B, n, C, out["X_next"],
                               stream)
        e[3].record(stream)
    barrier()
    return {k: [evs[s][i].elapsed_time(evs[s][i + 1]) for s in range(steps)]
            for i, k in enumerate(KERNELS)}


def gemm_after(mhc, stream, steps, warmup, wl, X, phi_t, F_out, bias, out) -> dict:
    """Median CUDA-event time (µs) of the GEMM entry point (steps 1-3) right after
    each predecessor, issued back to back on one stream: what the L2 holds when the
    GEMM starts (clean lines, or an earlier kernel's output still dirty) shows in
    its time."""
    import torch

    B, n, C = wl.B, wl.n, wl.C
    rd = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    wr = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")

    def gemm():
        mhc.mhc_gemm_rms_coeffs(X, phi_t, wl.alpha_pre, wl.alpha_post, wl.alpha_res, bias,
                                wl.iters, B, n, C, out["Y"], out["r"], out["H_pre"],
                                out["H_post"], out["H_res"], out["ws"], stream)

    def post():
        mhc.mhc_post_res_apply(X, F_out, out["H_res"], out["H_post"], B, n, C, out["X_next"],
                               stream)

    def pre():
        mhc.mhc_pre_apply(X, out["H_pre"], B, n, C, out["F_pre"], stream)

    def read512():
        rd.sum(dtype=torch.int64)

    def write512():
        wr.fill_(3)

    cases = {"gemm": [gemm], "post_res_apply": [post], "pre_apply": [pre],
             "post_res_apply, then a 512 MB read": [post, read512],
             "a 512 MB read": [read512], "a 512 MB write": [write512]}
    res = {}
    with torch.cuda.stream(stream):
        for label, before in cases.items():
            ts = []
            for it in range(warmup + steps):
                for f in before:
                    f()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                gemm()
                e1.record(stream)
                torch.cuda.synchronize()
                if it >= warmup:
                    ts.append(e0.elapsed_time(e1) * 1000.0)
            res[label] = statistics.median(ts)
    return res


def host_link_copy(h_X, h_F, h_out, X, F_out, out, stream):
    """One step's bytes over the host link with nothing else running: X and
    F_out host->device on `stream` while every output goes device->host on a
    second stream; returns the function that enqueues it."""
    import torch

    side = torch.cuda.Stream(device=X.device)

    def once():
        side.wait_stream(stream)
        with torch.cuda.stream(stream):
            X.copy_(h_X, non_blocking=True)
            F_out.copy_(h_F, non_blocking=True)
        with torch.cuda.stream(side):
            for k, v in h_out.items():
                v.copy_(out[k], non_blocking=True)
        stream.wait_stream(side)

    return once


def run_rmsnorm_gemm(args) -> int:
    """C = rmsnorm(A) @ B on one GPU: TFLOP/s of the fused kernel against the
    measured bf16 peak, beside cuBLAS's plain A @ B and PyTorch's
    rmsnorm-then-matmul of the same shape (context, not targets).  A, B
    ~N(0,1), N(0,0.02²) bf16, eps 1e-5; A is larger than L2 for the default
    shape, and every step reads it again."""
    import torch

    import gemm_rms_sinkhorn_gb300 as mhc
    import synth

    M, K, N = (int(v) for v in args.gemm.split(","))
    dev = torch.device("cuda", 0)
    to_dev = lambda bits: torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)
    A = to_dev(synth.normal_bf16((M, K), 51, 0))
    B_t = to_dev(synth.normal_bf16((N, K), 51, 2, 0.02))
    C = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    nbytes = mhc._lib.mhc_rmsnorm_gemm_workspace_bytes(M, K, N)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev) if nbytes else None
    stream = torch.cuda.current_stream(dev)
    flop = 2.0 * M * N * K

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    ours = timed(lambda: mhc.mhc_rmsnorm_gemm(A, B_t, M, K, N, 1e-5, C, ws, stream))
    cublas = timed(lambda: torch.matmul(A, B_t.t()))

    def torch_rms_mm():
        rstd = torch.rsqrt(A.float().pow(2).mean(-1, keepdim=True) + 1e-5)
        return torch.matmul((A.float() * rstd).to(torch.bfloat16), B_t.t())

    eager = timed(torch_rms_mm)
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, src = float(json.load(f)["bf16_tflops"]), "MEASURED_PEAKS.json bf16_tflops"
    except Exception:
        peak, src = 1900.0, "profiling-recipe fallback 1.9 PFLOP/s"
    tf = flop / (ours * 1e-3) / 1e12
    line = {"mode": "rmsnorm_gemm", "M": M, "K": K, "N": N, "eps": 1e-5, "steps": args.steps,
            "ms": ours, "tflops": tf,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                         "frac": tf / peak, "peak_source": src + " (of measured)"},
            "hbm_GBps": (2.0 * (M * K + N * K + M * N)) / (ours * 1e-3) / 1e9,
            "cublas_matmul_ms": cublas, "cublas_matmul_tflops": flop / (cublas * 1e-3) / 1e12,
            "torch_rmsnorm_then_matmul_ms": eager}
    print(json.dumps(line), flush=True)
    return 0


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-tokens", type=int, default=0,
                    help="tokens per step of the --impl reference arm (default 32 per host "
                         "core)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--clock-window", type=float, default=1.0,
                    help="seconds of identical load kept up for the clock samples")
    ap.add_argument("--path", default="auto", choices=["auto", "chain", "decode", "fused"],
                    help="forward path of each step: auto (mhc_forward's own choice) or one "
                         "forced through its test hook: chain (three kernels), decode (the "
                         "small-batch one-launch steps 1-4a), fused (the large-batch one-kernel "
                         "steps 1-4a)")
    ap.add_argument("--precision", default="bf16", choices=["bf16", "f32w", "e4m3"],
                    help="latency mode: f32w times mhc_forward_f32w (fp32 weight as split bf16 "
                         "pairs, fp32 F_out), e4m3 times mhc_forward_e4m3 (fp8 activations "
                         "and weight), instead of the bf16 forward")
    ap.add_argument("--tokens", type=int, default=None,
                    help="latency and kernels modes: the workload with this many tokens instead")
    ap.add_argument("--mode", default="full",
                    choices=["full", "kernels", "latency", "rmsnorm_gemm", "gemm_after"],
                    help="kernels: only the per-kernel loop (small runs for ncu captures); "
                         "gemm_after: the GEMM's event time after each predecessor "
                         "(another GEMM, the apply kernels, a 512 MB read or write); "
                         "latency: microseconds per mhc_forward (stream and CUDA graph); "
                         "rmsnorm_gemm: C = rmsnorm(A) @ B (Lazy Pre-Norm) on --gemm M,K,N")
    ap.add_argument("--gemm", default="16384,2048,2048",
                    help="rmsnorm_gemm mode: M,K,N")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)

    import synth

    wl = synth.WORKLOADS[args.workload]
    if args.tokens is not None:
        if args.mode not in ("latency", "kernels"):
            ap.error("--tokens only applies to --mode latency and --mode kernels")
        wl = wl.with_(name="%s_B%d" % (wl.name, args.tokens), B=args.tokens)
    if args.impl == "reference":
        return run_reference(args, wl)
    if args.mode == "rmsnorm_gemm":
        return run_rmsnorm_gemm(args)

    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist_mod

        dist = dist_mod
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    import gemm_rms_sinkhorn_gb300 as mhc

    B, n, C = wl.B, wl.n, wl.C
    inp = synth.make_inputs(wl, seed=rank)

    def to_dev_bf16(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

    X = to_dev_bf16(inp["X"])
    F_out = to_dev_bf16(inp["F_out"])
    phi_t = to_dev_bf16(inp["phi_t"])
    bias = torch.from_numpy(inp["bias"]).to(dev)
    out = mhc.alloc_outputs(B, n, C, dev)
    stream = torch.cuda.current_stream(dev)

    forward_call = {"auto": mhc.mhc_forward, "chain": mhc.mhc_testing_forward_chain,
                    "decode": mhc.mhc_testing_forward_decode,
                    "fused": mhc.mhc_testing_forward_fused}[args.path]
    if args.precision == "f32w":
        if args.mode != "latency":
            ap.error("--precision f32w only applies to --mode latency")
        # an fp32 weight (split once into bf16 pairs) and an fp32 F_out
        phi32 = torch.from_numpy(synth.normal_f32((wl.N, wl.K), rank, 2, wl.phi_std)).to(dev)
        phi_t = torch.empty(2 * wl.N, wl.K, dtype=torch.bfloat16, device=dev)
        mhc.mhc_split_phi(phi32, n, C, phi_t)
        F_out = torch.from_numpy(synth.normal_f32((B, C), rank, 1, wl.fout_std)).to(dev)
        forward_call = mhc.mhc_forward_f32w
    elif args.precision == "e4m3":
        if args.mode != "latency":
            ap.error("--precision e4m3 only applies to --mode latency")
        to8 = lambda a: torch.from_numpy(a).to(dev)
        X = to8(synth.normal_e4m3((B, wl.K), rank, 0, 1.0))
        phi_t = to8(synth.normal_e4m3((wl.N, wl.K), rank, 2, wl.phi_std))
        F_out = to8(synth.normal_e4m3((B, C), rank, 1, wl.fout_std))
        out["F_pre"] = torch.empty(B, C, dtype=torch.uint8, device=dev)
        out["X_next"] = torch.empty(B, wl.K, dtype=torch.uint8, device=dev)
        forward_call = mhc.mhc_forward_e4m3

    def step(on_stream=None):
        forward_call(X, phi_t, F_out, wl.alpha_pre, wl.alpha_post, wl.alpha_res, bias,
                     wl.iters, B, n, C, out["Y"], out["r"], out["H_pre"], out["H_post"],
                     out["H_res"], out["F_pre"], out["X_next"], out["ws"],
                     on_stream if on_stream is not None else stream)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    sampler = ClockSampler(gpu_id)
    time.sleep(0.3)

    if args.mode == "latency":
        sampler.stop()
        res = forward_latency(mhc, step, stream, barrier, args.steps, args.warmup)
        alg = sum(algorithmic_bytes(B, n, C, args.precision).values())
        if rank == 0:
            print(json.dumps({"mode": "latency", "workload": wl.name, "B": B, "n": n, "C": C,
                              "path": args.path, "precision": args.precision, **res,
                              "algorithmic_bytes": alg,
                              "GBps_graph": alg / (res["us_per_forward_graph"] * 1e-6) / 1e9}),
                  flush=True)
        return 0

    if args.mode == "gemm_after":
        print(json.dumps({"mode": "gemm_after", "workload": wl.name,
                          "us": gemm_after(mhc, stream, args.steps, args.warmup, wl, X, phi_t,
                                           F_out, bias, out)}), flush=True)
        sampler.stop()
        return 0

    if args.mode == "kernels":
        # warm up the three entry points timed below (mhc_forward may take
        # another path at this batch)
        if args.warmup > 0:
            per_kernel_times(mhc, stream, barrier, args.warmup, wl, X, phi_t, F_out, bias, out)
        ms = per_kernel_times(mhc, stream, barrier, args.steps, wl, X, phi_t, F_out, bias, out)
        sampler.stop()
        if dist is not None:
            dist.destroy_process_group()
        if rank == 0:
            print(json.dumps({"mode": "kernels", "workload": wl.name, "ms": ms}), flush=True)
        return 0

    # ---- timed region: K whole forward steps
    for _ in range(args.warmup):
        step()
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_host0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    barrier()
    ms_total = ev0.elapsed_time(ev1)
    # keep the same load up for ~1 s when the timed region is short, so the
    # clock samples describe the loaded state of the timed steps
    t_host1 = time.time()
    extra_until = t_host0 + args.clock_window
    while time.time() < extra_until:
        for _ in range(20):
            step()
        torch.cuda.synchronize(dev)
    t_host2 = time.time()
    ms_total = max_over_ranks(ms_total, dist, dev)
    ms_step = ms_total / args.steps
    value = tokens_per_second(B, world, args.steps, ms_total)

    # ---- per-kernel CUDA-event times over the same steps (same stream)
    runs = per_kernel_runs(mhc, stream, barrier, args.steps, wl, X, phi_t, F_out, bias, out)
    per_kernel_ms = {k: statistics.mean(v) for k, v in runs.items()}
    sampler.stop()
    status = mhc.mhc_device_status()
    if status != mhc.MHC_OK:
        raise RuntimeError("device status %s after the timed steps" % mhc.mhc_status_str(status))

    algo = kernel_bytes(B, n, C)
    peak, peak_src = measured_peaks()
    dom = max(KERNELS, key=lambda k: per_kernel_ms[k])
    achieved = algo[dom] / (per_kernel_ms[dom] / 1e3) / 1e9
    total_bytes = sum(algorithmic_bytes(B, n, C).values())  # the steps' compulsory bytes
    # "ms" is the mean over the steps (the roofline's average launch); the
    # median and the fastest step are there beside it
    kernels_json = {k: {"ms": per_kernel_ms[k], "median_ms": statistics.median(runs[k]),
                        "min_ms": min(runs[k]), "algorithmic_bytes": algo[k],
                        "GBps": algo[k] / (per_kernel_ms[k] / 1e3) / 1e9,
                        "frac": algo[k] / (per_kernel_ms[k] / 1e3) / 1e9 / peak}
                    for k in KERNELS}

    # ---- end to end through the public API with pinned host buffers: the
    # host-buffer forward copies each step's inputs (X, F_out) to the device and
    # every output back, overlapped with the compute chunk by chunk; the
    # weights (phi_t, b) stay resident on the device as in a model
    h_X = torch.empty(X.shape, dtype=X.dtype, pin_memory=True)
    h_X.copy_(X)
    h_F = torch.empty(F_out.shape, dtype=F_out.dtype, pin_memory=True)
    h_F.copy_(F_out)
    h_out = mhc.alloc_host_outputs(B, n, C, pin=True)
    scratch = mhc.host_scratch(B, n, C, dev)

    def e2e_step():
        mhc.mhc_forward_host(h_X, phi_t, h_F, wl.alpha_pre, wl.alpha_post, wl.alpha_res, bias,
                             wl.iters, B, n, C, h_out["Y"], h_out["r"], h_out["H_pre"],
                             h_out["H_post"], h_out["H_res"], h_out["F_pre"], h_out["X_next"],
                             scratch, stream)

    h2d = sum(t.numel() * t.element_size() for t in (h_X, h_F))
    d2h = sum(t.numel() * t.element_size() for t in h_out.values())
    link_once = host_link_copy(h_X, h_F, h_out, X, F_out, out, stream)
    for _ in range(2):
        e2e_step()
        link_once()
    barrier()
    # the e2e steps and, after each, the same bytes as plain copies (the host
    # link's own bound; the link is shared with the node's other work, so the
    # two are interleaved rather than taken one after the other)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.e2e_steps)]
    for e in ev:
        e[0].record(stream)
        e2e_step()
        e[1].record(stream)
        link_once()
        e[2].record(stream)
    barrier()
    e2e_ms = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in ev), dist, dev) / args.e2e_steps
    e2e_value = tokens_per_second(B, world, 1, e2e_ms)
    link_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / args.e2e_steps

    # ---- CPU baseline: the fp64 oracle on the host cores (rank 0 only)
    cpu = None
    if rank == 0 and world == 1:
        rate1, tokens1, secs1 = cpu_oracle_rate(wl, inp, args.cpu_budget)
        cores = os.cpu_count() or 1
        pool = OracleOnAllCores(wl, inp, cores)
        # all cores: as many tokens as the 1-core leg's budget covers on every core
        tok_all = min(B, max(cores * 32, int(rate1 * args.cpu_budget * cores / 2)))
        rate_all, secs_all = pool.rate(tok_all)
        pool.close()
        cpu = {"value": rate_all, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": "first %d tokens of B=%d n=%d C=%d, fp64 oracle forward split by "
                         "token range over %d host threads, %.1f s" % (
                             tok_all, B, n, C, cores, secs_all),
               "cpu": cpu_model(), "host_cores": os.cpu_count(),
               "single_core": {"value": rate1, "unit": "tokens/s", "cores": 1,
                               "sample": "first %d tokens, one thread, %.1f s" % (tokens1,
                                                                                  secs1)}}

    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return 0
    clocks = sampler.summary(t_host0, max(t_host1, t_host2))
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded counter-based generator; X rows N(0, s^2), s log-uniform"
                " in [0.1, 10])",
        "config": workload_config(wl, world),
        "hbm_GBps_forward": total_bytes / (ms_step / 1e3) / 1e9,
        "roofline_forward": {"algorithmic_bytes": total_bytes, "peak": peak,
                             "frac": total_bytes / (ms_step / 1e3) / 1e9 / peak},
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "traffic": stored_traffic(dom),
                     "algorithmic_bytes": algo[dom], "peak_source": peak_src},
        "kernels": kernels_json,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "link_copy_ms_per_step": link_ms,
                "link_frac": link_ms / e2e_ms if e2e_ms > 0 else None},
        "gpu_launches": LAUNCHES_PER_STEP * args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
