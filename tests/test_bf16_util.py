"""Pins of the tests' bf16 rounding helper against the definition of bf16
(1 sign, 8 exponent, 7 fraction bits; round to nearest, ties to even)."""
import numpy as np

from bf16_util import bf16_bits_to_f32, round_to_bf16, to_bf16_bits


def test_exact_values_keep_their_bits():
    v = np.array([0.0, 1.0, -2.0, 0.5, 3.0, 1.0 + 2.0 ** -7, 65280.0], dtype=np.float32)
    b = to_bf16_bits(v)
    assert (bf16_bits_to_f32(b) == v).all()
    assert b[1] == 0x3F80 and b[2] == 0xC000


def test_round_to_nearest_and_ties_to_even():
    one = 1.0
    ulp = 2.0 ** -7                     # bf16 spacing in [1, 2)
    cases = [
        (one + 0.25 * ulp, one),        # below half: down
        (one + 0.75 * ulp, one + ulp),  # above half: up
        (one + 0.5 * ulp, one),         # tie, 1.0 has an even fraction: stays
        (one + 1.5 * ulp, one + 2 * ulp),   # tie, odd neighbour below: up to even
        (-(one + 0.75 * ulp), -(one + ulp)),
    ]
    x = np.array([c[0] for c in cases], dtype=np.float32)
    want = np.array([c[1] for c in cases], dtype=np.float32)
    assert (round_to_bf16(x) == want).all()


def test_relative_rounding_error_is_at_most_half_an_ulp():
    # 8 significant bits: unit roundoff 2^-8
    rng = np.random.default_rng(5)
    x = rng.standard_normal(100000).astype(np.float32) * 10.0 ** rng.integers(-3, 4, 100000)
    r = round_to_bf16(x).astype(np.float64)
    rel = np.abs(r - x) / np.abs(x)
    assert rel.max() <= 2.0 ** -8
    assert rel.max() > 2.0 ** -9   # and the bound is reached in practice
    # a bf16 value has at most 8 significant bits
    m, _ = np.frexp(r)
    assert (np.abs(m * 2 ** 8 - np.round(m * 2 ** 8)) == 0).all()
