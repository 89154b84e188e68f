"""Host side of the seeded input generator: determinism, offsets, rounding, distribution."""
import numpy as np

import synth


def test_deterministic_and_offset_consistent():
    a = synth.host_bits(synth.F32, (1000,), 7, 3, 0.0, 1.0)
    b = synth.host_bits(synth.F32, (1000,), 7, 3, 0.0, 1.0)
    np.testing.assert_array_equal(a, b)
    c = synth.host_bits(synth.F32, (400,), 7, 3, 0.0, 1.0, offset=600)
    np.testing.assert_array_equal(a[600:], c)
    d = synth.host_bits(synth.F32, (1000,), 7, 4, 0.0, 1.0)
    assert not np.array_equal(a, d)


def test_distribution_moments_and_bound():
    z = synth.host_f64(synth.F32, (1 << 20,), 11, 1, 0.0, 1.0)
    assert abs(z.mean()) < 5e-3 and abs(z.std() - 1) < 5e-3
    assert np.abs(z).max() <= 6.0
    # Irwin-Hall values are multiples of 2^-16 (exact in f32)
    assert np.all(z * 65536 == np.round(z * 65536))


def test_bf16_is_rne_of_f32():
    f = synth.host_bits(synth.F32, (50000,), 5, 9, 0.0, 0.02)
    b = synth.host_bits(synth.BF16, (50000,), 5, 9, 0.0, 0.02)
    u = f.view(np.uint32).astype(np.uint64)
    rne = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    np.testing.assert_array_equal(b, rne)
    np.testing.assert_array_equal(synth.bf16_bits_to_f64(b), synth.host_f64(synth.BF16, (50000,), 5, 9, 0.0, 0.02))


def test_constant_fill():
    g = synth.host_f64(synth.BF16, (64,), 1, 2, 1.0, 0.0)
    assert np.all(g == 1.0)
