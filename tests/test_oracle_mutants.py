"""Planted mistakes in a copy of the oracle must each break at least one pin.

Each mutant is a one-line edit of ``oracle/mhc_oracle.c`` (a dropped term, a
wrong sign, index or operand order, an off-by-one), compiled on the CPU into a
temporary library and swapped in for the real one while the pins run.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "mhc_oracle.c")

MUTANTS = {
    "bias dropped": ("* Y[b * N + k] / r[b] + bias[k];", "* Y[b * N + k] / r[b];"),
    "r multiplies": ("* Y[b * N + k] / r[b] + bias[k];", "* Y[b * N + k] * r[b] + bias[k];"),
    "alpha segments swapped": ("k < n ? a_pre : (k < 2 * n ? a_post : a_res)",
                               "k < n ? a_post : (k < 2 * n ? a_pre : a_res)"),
    "rms over C": ("r[b] = sqrt(ss / (double)K);", "r[b] = sqrt(ss / (double)C);"),
    "rms without sqrt": ("r[b] = sqrt(ss / (double)K);", "r[b] = ss / (double)K;"),
    "phi transposed": ("oracle_bf16_to_f64(phi[q * N + k])", "oracle_bf16_to_f64(phi[k * K + q])"),
    "sigmoid sign": ("H_pre[b * n + i] = 1.0 / (1.0 + exp(-h[i]));",
                     "H_pre[b * n + i] = 1.0 / (1.0 + exp(h[i]));"),
    "post factor 1": ("H_post[b * n + i] = 2.0 / (1.0 + exp(-h[n + i]));",
                      "H_post[b * n + i] = 1.0 / (1.0 + exp(-h[n + i]));"),
    "post reads pre": ("2.0 / (1.0 + exp(-h[n + i]))", "2.0 / (1.0 + exp(-h[i]))"),
    "no exp": ("H_res[i] = exp(Ht_res[i]);", "H_res[i] = Ht_res[i];"),
    "one extra iteration": ("for (int t = 0; t < iters; ++t)", "for (int t = 0; t <= iters; ++t)"),
    "column step dropped": ("                H_res[i * n + j] /= s;\n        }\n    }\n}",
                            "                H_res[i * n + j] /= 1.0;\n        }\n    }\n}"),
    "column then row": ("                s += H_res[i * n + j];\n            for (int j = 0; j < n; ++j)\n                H_res[i * n + j] /= s;",
                        "                s += H_res[j * n + i];\n            for (int j = 0; j < n; ++j)\n                H_res[j * n + i] /= s;"),
    "pre stream layout": ("H_pre[b * n + i] * oracle_bf16_to_f64(X[b * K + (int64_t)i * C + c])",
                          "H_pre[b * n + i] * oracle_bf16_to_f64(X[b * K + c * n + i])"),
    "H_res transposed": ("x_res += h[i * n + j]", "x_res += h[j * n + i]"),
    "post term dropped": ("X_next[b * K + (int64_t)i * C + c] = x_res + x_post;",
                          "X_next[b * K + (int64_t)i * C + c] = x_res;"),
    "F_out index": ("oracle_bf16_to_f64(F_out[b * C + c])", "oracle_bf16_to_f64(F_out[c])"),
    "forward skips pre": ("    oracle_pre_apply(X, H_pre, B, n, C, F_pre);\n", ""),
    "rmsnorm drops eps": ("1.0 / sqrt(ss / (double)K + eps);", "1.0 / sqrt(ss / (double)K);"),
    "rmsnorm sum not mean": ("1.0 / sqrt(ss / (double)K + eps);", "1.0 / sqrt(ss + eps);"),
    "rmsnorm B transposed": ("oracle_bf16_to_f64(Bm[q * N + k])", "oracle_bf16_to_f64(Bm[k * K + q])"),
    "f64 phi rounded to float": ("acc += oracle_bf16_to_f64(X[b * K + q]) * phi[q * N + k];",
                                 "acc += oracle_bf16_to_f64(X[b * K + q]) * (double)(float)(phi[q * N + k] * 1.0009765625);"),
    "f64 F_out index": ("H_post[b * n + i] * F_out[b * C + c];", "H_post[b * n + i] * F_out[c];"),
    "e4m3 exponent bias": ("return s * ldexp(1.0 + m / 8.0, e - 7);", "return s * ldexp(1.0 + m / 8.0, e - 8);"),
    "e4m3 subnormal scale": ("return s * ldexp((double)m, -9);", "return s * ldexp((double)m, -10);"),
    "e4m3 F_pre drops a stream": ("for (int i = 0; i < n; ++i) f += H_pre[b * n + i]", "for (int i = 1; i < n; ++i) f += H_pre[b * n + i]"),
}


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation anchor missing for %r" % name
    mutated = src.replace(old, new, 1)
    d = tmp_path / name.replace(" ", "_")
    d.mkdir()
    (d / "mhc_oracle.c").write_text(mutated)
    hdr = os.path.join(os.path.dirname(SRC), "mhc_oracle.h")
    (d / "mhc_oracle.h").write_text(open(hdr).read())
    so = d / "libmut.so"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-shared", "-fPIC",
                           "-o", str(so), str(d / "mhc_oracle.c"), "-lm"])
    return oracle._configure(ctypes.CDLL(str(so)))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    lib = _build_mutant(tmp_path, name, old, new)
    saved = oracle._load()
    failed = []
    try:
        oracle._lib = lib
        for pin in oracle_pins.ALL_PINS:
            try:
                pin()
            except (AssertionError, FloatingPointError, ValueError, ZeroDivisionError):
                failed.append(pin.__name__)
    finally:
        oracle._lib = saved
    assert failed, "no pin catches the planted mistake %r" % name


def test_pins_pass_on_the_real_oracle():
    for pin in oracle_pins.ALL_PINS:
        pin()
