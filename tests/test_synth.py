"""The seeded input generator: determinism, prefix property, distributions (CPU)."""
import numpy as np

import synth
from synth import WORKLOADS, make_inputs


def test_thread_count_independent():
    a = synth.normal_bf16((300, 1000), 0, 0, 1.0, nthreads=1)
    b = synth.normal_bf16((300, 1000), 0, 0, 1.0, nthreads=7)
    assert np.array_equal(a, b)


def test_prefix_rows_match_full_size():
    wl = WORKLOADS["tiny"]
    full = make_inputs(wl, seed=0)
    part = make_inputs(wl, seed=0, rows=5)
    assert np.array_equal(full["X"][:5], part["X"])
    assert np.array_equal(full["F_out"][:5], part["F_out"])
    assert np.array_equal(full["phi_t"], part["phi_t"])
    assert np.array_equal(full["bias"], part["bias"])


def test_streams_differ_by_seed_and_tensor():
    a = synth.normal_f32(1000, 0, 0)
    assert not np.array_equal(a, synth.normal_f32(1000, 1, 0))
    assert not np.array_equal(a, synth.normal_f32(1000, 0, 1))


def test_normal_moments():
    x = synth.bf16_bits_to_f32(synth.normal_bf16(400000, 0, 0, 0.02)).astype(np.float64)
    assert abs(x.mean()) < 1e-4 and abs(x.std() - 0.02) < 2e-4


def test_rowscale_sigma_range():
    X = synth.bf16_bits_to_f32(synth.rowscale_normal_bf16(200, 4096, 0, 0, 4)).astype(np.float64)
    s = X.std(axis=1)
    assert s.min() > 0.08 and s.max() < 12 and s.max() / s.min() > 20


def test_student_t_heavy_tail():
    x = synth.bf16_bits_to_f32(synth.student_t_bf16(200000, 0, 0, 3)).astype(np.float64)
    # t_3 has variance 3 and far heavier tails than a normal
    assert 2.0 < x.var() < 5.0 and np.abs(x).max() > 15


def test_int_range_exact():
    v = synth.bf16_bits_to_f32(synth.int_bf16(10000, 0, 0, -2, 2))
    assert set(np.unique(v).tolist()) == {-2.0, -1.0, 0.0, 1.0, 2.0}


def test_bf16_rounding_round_trip():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -3.5, 1e-40], dtype=np.float32)
    got = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(x))
    # ties to even: 1+2^-8 -> 1.0, 1+3*2^-8 -> 1+2^-6
    assert got[0] == 1.0 and got[1] == 1.0 and got[2] == 1.0 + 2 ** -6 and got[3] == -3.5


def test_e4m3_codec_round_trip_and_ties():
    import numpy as np
    import synth
    codes = np.arange(256, dtype=np.uint8)
    vals = synth.e4m3_bits_to_f32(codes)
    finite = ~np.isnan(vals)
    assert np.array_equal(synth.f32_to_e4m3_bits(vals[finite]), codes[finite])
    assert vals[0x38] == 1.0 and vals[0x7E] == 448.0 and vals[0x01] == 2.0 ** -9
    assert vals[0x08] == 2.0 ** -6 and vals[0xB8] == -1.0 and np.isnan(vals[0x7F])
    # midpoints between neighbouring positive codes go to the even code
    pos = vals[:0x7F].astype(np.float64)
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    got = synth.f32_to_e4m3_bits(mids)
    lo = np.arange(0, 0x7E)
    want = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(got, want.astype(np.uint8))
    # saturation and NaN
    assert synth.f32_to_e4m3_bits(np.array([1e6, -500.0, np.inf], np.float32)).tolist() == [0x7E, 0xFE, 0x7E]
    assert synth.f32_to_e4m3_bits(np.array([np.nan], np.float32))[0] == 0x7F
