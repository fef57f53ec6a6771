"""The seeded input generator: determinism, distribution, bf16 rounding."""
import numpy as np

from linear_recurrent_sequence_gb300 import synth


def test_deterministic_and_distinct_streams():
    a = synth.normal(1003, synth.STREAMS["q"], (1000,))
    b = synth.normal(1003, synth.STREAMS["q"], (1000,))
    c = synth.normal(1003, synth.STREAMS["k"], (1000,))
    assert np.array_equal(a, b) and not np.array_equal(a, c)


def test_standard_normal_moments():
    x = synth.normal(7, 1, (200000,))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert abs(((x - x.mean()) ** 3).mean()) < 0.03


def test_bf16_round_to_nearest_even():
    f = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5, 1.0 + 2.0 ** -9],
                 dtype=np.float32)
    bits = synth.f32_to_bf16_bits(f)
    # 1+2^-8 is a tie -> even (1.0); 1+3*2^-8 is a tie -> even (1+2^-6 pattern 0x3F82)
    assert list(bits) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x3F80]
    assert np.array_equal(synth.bf16_bits_to_f64(bits)[[0, 3]], [1.0, -2.5])


def test_tensor_values_are_exact_widening():
    bits, x64 = synth.tensor(1002, "v", (3, 5), "bf16")
    assert bits.dtype == np.uint16 and x64.dtype == np.float64
    back = synth.f32_to_bf16_bits(x64.astype(np.float32))
    assert np.array_equal(back, bits)


def test_head_gammas():
    g = synth.head_gammas(3)
    assert np.array_equal(g, [1 - 2.0 ** -5, 1 - 2.0 ** -6, 1 - 2.0 ** -7])
