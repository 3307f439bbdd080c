"""Pins of the oracle's bf16 rounding (oracle/numerics.py).

bf16 keeps float32's sign and exponent and 7 stored mantissa bits; rounding
is to nearest, ties to even.  Each check below fixes a value the definition
of the format decides, or compares against a rounding computed a different
way (integer arithmetic on float32 bit patterns, and torch's own cast).
"""
import numpy as np
import pytest

from oracle.numerics import round_bf16

ULP1 = 2.0 ** -7  # spacing of bf16 values in [1, 2)


@pytest.mark.parametrize("x, want", [
    (1.0, 1.0),
    (1.0 + 2.0 ** -8, 1.0),                       # halfway 1 .. 1+2^-7: tie to the even mantissa (0)
    (1.0 + 3 * 2.0 ** -8, 1.0 + 2 * ULP1),        # halfway 1+2^-7 .. 1+2^-6: tie to the even mantissa (2)
    (1.0 + 3 * 2.0 ** -9, 1.0 + ULP1),            # 0.75 ulp above 1: nearest is 1+2^-7
    (1.0 + 2.0 ** -9, 1.0),                       # 0.25 ulp: down
    (-(1.0 + 2.0 ** -8), -1.0),                   # negative tie
    (-(1.0 + 3 * 2.0 ** -8), -(1.0 + 2 * ULP1)),
    (3.0 + 2.0 ** -7, 3.0),                       # [2, 4): spacing 2^-6, tie -> even (3.0 = 1.1000000b)
    (0.0, 0.0),
    (2.0 ** 127 * (2 - 2.0 ** -7), 2.0 ** 127 * (2 - 2.0 ** -7)),   # largest finite
    (2.0 ** 127 * (2 - 2.0 ** -8) * (1 - 2.0 ** -30), 2.0 ** 127 * (2 - 2.0 ** -7)),  # just below the tie
    (2.0 ** 127 * (2 - 2.0 ** -8), np.inf),       # tie between max (odd mantissa) and 2^128: overflow
    (-(2.0 ** 127) * 2.0, -np.inf),
    (2.0 ** -126, 2.0 ** -126),                   # smallest normal
    (2.0 ** -133, 2.0 ** -133),                   # smallest subnormal
    (3 * 2.0 ** -134, 2 * 2.0 ** -133),           # subnormal tie 1.5 quanta -> 2 (even)
    (2.0 ** -134, 0.0),                           # half the smallest subnormal: tie to zero
    (2.0 ** -134 * 1.001, 2.0 ** -133),
    (127.5 * 2.0 ** -133, 128 * 2.0 ** -133),     # subnormal tie rounding up into the normal range
])
def test_round_bf16_exact_values(x, want):
    got = float(round_bf16(np.float64(x)))
    assert got == want, (x, got, want)


def _bits_round(f32: np.ndarray) -> np.ndarray:
    """bf16 rounding of float32 values by integer arithmetic on their bit
    patterns: add 0x7FFF plus the lowest kept bit, then clear the low 16
    bits (carries into the exponent handle mantissa overflow and infinity)."""
    u = f32.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def test_round_bf16_matches_bit_level_rounding():
    rng = np.random.default_rng(11)
    parts = [rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
             rng.standard_normal(5000) * 2.0 ** -130,                # subnormal range
             (1 + rng.integers(0, 2 ** 16, 5000) / 2 ** 16) * 2.0 ** rng.integers(-20, 20, 5000)]
    x = np.concatenate(parts).astype(np.float32)   # float32-exact inputs: no double rounding
    x = x[np.isfinite(x)]
    np.testing.assert_array_equal(round_bf16(x.astype(np.float64)), _bits_round(x))


def test_round_bf16_matches_torch_cast():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(12)
    x = (rng.standard_normal(50000) * 10.0 ** rng.integers(-8, 8, 50000)).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(round_bf16(x.astype(np.float64)), want)


def test_round_bf16_keeps_8_significant_bits():
    # every output is a multiple of its own 2^(e-8) and within half a spacing of the input
    rng = np.random.default_rng(13)
    x = rng.standard_normal(10000) * 100
    r = round_bf16(x)
    m, e = np.frexp(r)
    assert np.all(np.ldexp(m, 8) == np.rint(np.ldexp(m, 8)))
    _, ex = np.frexp(x)
    assert np.all(np.abs(r - x) <= np.ldexp(1.0, ex - 9))
