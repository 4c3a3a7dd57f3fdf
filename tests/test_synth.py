"""The seeded input generator (CPU side; the device twin is checked in test_parity_small)."""
import numpy as np

import synth


def test_deterministic_and_position_addressable():
    a = synth.normal_bf16(1, synth.K, 2, 3, 0, range(10, 20), 4, 64)
    b = synth.normal_bf16(1, synth.K, 2, 3, 0, [15], 4, 64)
    assert a.shape == (10, 4, 64) and a.dtype == np.uint16
    assert np.array_equal(a[5], b[0])
    assert np.array_equal(a, synth.normal_bf16(1, synth.K, 2, 3, 0, range(10, 20), 4, 64))


def test_streams_differ():
    base = synth.normal_bf16(0, synth.Q, 0, 0, 0, range(4), 2, 32)
    for args in [(1, synth.Q, 0, 0, 0), (0, synth.K, 0, 0, 0), (0, synth.Q, 1, 0, 0),
                 (0, synth.Q, 0, 1, 0), (0, synth.Q, 0, 0, 1)]:
        other = synth.normal_bf16(*args, range(4), 2, 32)
        assert np.mean(other == base) < 0.05


def test_moments_close_to_standard_normal():
    x = synth.bf16_to_f32(synth.normal_bf16(3, synth.V, 0, 0, 0, range(4096), 8, 128))
    x = x.astype(np.float64).ravel()
    assert abs(x.mean()) < 5e-3
    assert abs(x.std() - 1.0) < 5e-3
    assert np.abs(x).max() <= 6.0
    # Irwin-Hall(12) kurtosis is 3 - 0.1 = 2.9
    kurt = np.mean(x ** 4) / np.mean(x ** 2) ** 2
    assert 2.85 < kurt < 2.95


def test_values_are_bf16_roundings_of_multiples_of_2_pow_minus_16():
    x = synth.bf16_to_f32(synth.normal_bf16(5, synth.K, 0, 0, 0, range(64), 2, 64))
    assert np.all(np.isfinite(x))
    # every value is a bf16 number (low 16 bits of the float32 pattern are zero)
    assert np.all((x.view(np.uint32) & 0xFFFF) == 0)
