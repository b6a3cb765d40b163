"""Workload recipes: shapes and input distributions of the mHC forward cases.

Shapes follow the mHC page ("mHC 算法分析 & cutile 高效实现", §2 and §5: B tokens,
expansion n, hidden size C, K = n·C, N = n² + 2n).  Distributions are synthetic
stand-ins (no dataset or trained weights are involved).  Tensor ids used with
the counter-based generator: X=0, F_out=1, φ=2, bias=3, per-row σ=4.
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    n: int
    C: int
    iters: int = 20
    alpha_pre: float = 0.01
    alpha_post: float = 0.01
    alpha_res: float = 0.01
    x_kind: str = "normal"  # "normal" | "rowscale" | "student_t3"
    phi_std: float = 0.02
    bias_std: float = 0.1
    fout_std: float = 1.0

    @property
    def K(self) -> int:
        return self.n * self.C

    @property
    def N(self) -> int:
        return self.n * self.n + 2 * self.n

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    # B=64 tokens, n=4, C=256: the small case the oracle finishes at once
    "tiny": Workload("tiny", B=64, n=4, C=256),
    # 7B-width: B=4096, n=4, C=4096 (X 128 MiB bf16)
    "7b": Workload("7b", B=4096, n=4, C=4096),
    # prefill: B=16384, n=4, C=7168; row scales log-uniform in [0.1, 10]
    "prefill": Workload("prefill", B=16384, n=4, C=7168, x_kind="rowscale"),
    # decode shapes, latency bound
    "decode1": Workload("decode1", B=1, n=4, C=7168),
    "decode8": Workload("decode8", B=8, n=4, C=7168),
    "decode32": Workload("decode32", B=32, n=4, C=7168),
    "decode128": Workload("decode128", B=128, n=4, C=7168),
    # wider expansion: n=8 (N=80, 8x8 Sinkhorn), heavy-tailed X, larger bias
    "wider": Workload("wider", B=8192, n=8, C=4096, x_kind="student_t3", bias_std=0.5),
    "wider_it5": Workload("wider_it5", B=8192, n=8, C=4096, x_kind="student_t3",
                          bias_std=0.5, iters=5),
    "wider_it50": Workload("wider_it50", B=8192, n=8, C=4096, x_kind="student_t3",
                           bias_std=0.5, iters=50),
}


def make_inputs(wl: Workload, seed: int = 0, rows: int | None = None, nthreads: int = 0,
                parts=("X", "F_out", "phi_t", "bias")):
    """Generate the inputs of ``wl`` (first ``rows`` tokens if given).

    Returns a dict of numpy arrays: X [B, n*C] bf16 bits, F_out [B, C] bf16
    bits, phi_t [N, K] bf16 bits (φ transposed, K contiguous) and bias [N]
    float32.  The first ``rows`` tokens equal the first rows of the full-size
    arrays, because every element is a function of its index only.
    """
    from . import (int_bf16, normal_bf16, normal_f32, rowscale_normal_bf16,  # noqa: F401
                   student_t_bf16)

    B = wl.B if rows is None else rows
    out = {}
    if "X" in parts:
        if wl.x_kind == "normal":
            out["X"] = normal_bf16((B, wl.K), seed, 0, 1.0, nthreads)
        elif wl.x_kind == "rowscale":
            out["X"] = rowscale_normal_bf16(B, wl.K, seed, 0, 4, -1.0, 1.0, nthreads)
        elif wl.x_kind == "student_t3":
            out["X"] = student_t_bf16((B, wl.K), seed, 0, 3, 1.0, nthreads)
        else:
            raise ValueError(wl.x_kind)
    if "F_out" in parts:
        out["F_out"] = normal_bf16((B, wl.C), seed, 1, wl.fout_std, nthreads)
    if "phi_t" in parts:
        out["phi_t"] = normal_bf16((wl.N, wl.K), seed, 2, wl.phi_std, nthreads)
    if "bias" in parts:
        out["bias"] = normal_f32((wl.N,), seed, 3, wl.bias_std, nthreads)
    return out
