"""Helpers of the GPU parity tests: device transfers and the tolerance checks.

Tolerances (stated for the mHC forward this library implements):
  H_pre, H_post, H_res   |Δ| <= 2e-3 absolute
  r                      |Δr| / r <= 1e-3
  F_pre, X_next (bf16)   |Δ| <= 2^-7·|ref| + 1e-3 per element
  Y (fp32, no stated bound; derived from fp32 accumulation of K exact bf16
  products): |ΔY| <= 1e-5·Σ_q|X[b,q]·φ[q,k]| + 1e-6, far above the typical
  sqrt(K)·2^-24 rounding and far below the effect of a dropped 64-wide K block.
"""
import concurrent.futures
import os

import numpy as np
import torch

import synth

H_TOL = 2e-3
R_REL = 1e-3
BF16_REL = 2.0 ** -7
BF16_ABS = 1e-3
Y_REL = 1e-5


def cuda_ok() -> bool:
    return torch.cuda.is_available()


def dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(device)


def dev_f32(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def host64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def phi_KN(phi_t: np.ndarray) -> np.ndarray:
    """φ in its mathematical [K, N] orientation from the ABI's φᵀ [N, K]."""
    return np.ascontiguousarray(phi_t.T)


def f64(bits: np.ndarray) -> np.ndarray:
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def assert_abs(got, ref, tol, what):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "%s: non-finite output" % what
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    assert err <= tol, "%s: max |diff| %.3e > %.1e" % (what, err, tol)
    return err


def assert_rel(got, ref, tol, what):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    err = float(np.max(np.abs(got - ref) / np.abs(ref))) if got.size else 0.0
    assert err <= tol, "%s: max rel diff %.3e > %.1e" % (what, err, tol)
    return err


def assert_bf16_close(got, ref, what):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "%s: non-finite output" % what
    excess = np.abs(got - ref) - (BF16_REL * np.abs(ref) + BF16_ABS)
    worst = float(np.max(excess)) if got.size else -1.0
    assert worst <= 0.0, "%s: %d elements outside 2^-7|ref|+1e-3 (worst excess %.3e)" % (
        what, int(np.sum(excess > 0)), worst)


def assert_Y_close(got, ref, X_bits, phi_t_bits, what="Y"):
    absX = np.abs(f64(X_bits))
    absW = np.abs(f64(phi_t_bits))  # [N, K]
    bound = Y_REL * (absX @ absW.T) + 1e-6
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert got.shape == ref.shape
    excess = np.abs(got - ref) - bound
    assert np.max(excess) <= 0, "%s: worst excess %.3e" % (what, float(np.max(excess)))
    return float(np.max(np.abs(got - ref)))


def sample_rows(B: int, k: int = 48, seed: int = 0) -> np.ndarray:
    """Tile and edge rows plus random ones, sorted and unique."""
    fixed = {0, 1, 126, 127, 128, 129, B // 2, B - 129, B - 128, B - 2, B - 1}
    rng = np.random.default_rng(seed)
    extra = rng.choice(B, size=min(k, B), replace=False)
    rows = sorted(r for r in fixed.union(extra.tolist()) if 0 <= r < B)
    return np.array(rows, dtype=np.int64)


def for_all_rows(B: int, fn, chunk: int = 256, workers: int = 0) -> None:
    """Run ``fn(lo, hi)`` over every token range [lo, hi) of [0, B) on all host
    cores and re-raise the first failure.  Tokens are independent, so the
    single-threaded oracle can take a range at a time; its C call and numpy's
    array operations release the GIL."""
    workers = workers or os.cpu_count() or 4
    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        futs = [ex.submit(fn, lo, min(lo + chunk, B)) for lo in range(0, B, chunk)]
        for f in futs:
            f.result()


def host_outputs(out: dict) -> dict:
    """A forward's outputs on the host: fp32 ones widened to float64, bf16 ones
    kept as bit patterns (half the bytes of a float64 copy at full size)."""
    g = {k: host64(out[k]) for k in ("Y", "r", "H_pre", "H_post", "H_res")}
    for k in ("F_pre", "X_next"):
        g[k] = host_bits(out[k])
    return g
