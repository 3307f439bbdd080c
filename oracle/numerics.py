"""Number-format helpers of the oracle (test infrastructure only).

bf16 is float32's sign and 8-bit exponent with a 7-bit stored mantissa
(8 significant bits for normal values).  A bf16 model stores every layer
output in bf16; the oracle mirrors that storage with a direct
round-to-nearest-even from float64 (not through float32), written from the
definition of the format.
"""
import numpy as np

_BF16_MIN_NORMAL = 2.0 ** -126
_BF16_MAX = 2.0 ** 127 * (2 - 2.0 ** -7)


def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even.

    Normal range (|x| >= 2**-126): with x = m * 2**e and 0.5 <= |m| < 1
    (frexp), a bf16 value has 8 significant bits, i.e. m is a multiple of
    2**-8.  Below it the spacing is fixed at the subnormal quantum 2**-133
    (2**-126 spread over the 7 stored mantissa bits).  np.rint rounds half to
    even in both cases.  A result beyond bf16's largest finite value,
    (2 - 2**-7) * 2**127, is an overflow to infinity of the same sign.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    normal = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    sub = np.ldexp(np.rint(np.ldexp(x, 133)), -133)
    r = np.where(np.abs(x) < _BF16_MIN_NORMAL, sub, normal)
    r = np.where(np.abs(r) > _BF16_MAX, np.copysign(np.inf, r), r)
    return r


def round_f32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
