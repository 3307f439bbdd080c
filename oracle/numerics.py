"""Number-format helpers of the oracle (test infrastructure only).

bf16 is float32's sign and 8-bit exponent with a 7-bit stored mantissa
(8 significant bits).  A bf16 model stores every layer output in bf16; the
oracle mirrors that storage with a direct round-to-nearest-even from float64
(not through float32), written from the definition of the format.
"""
import numpy as np


def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even.

    With x = m * 2**e and 0.5 <= |m| < 1 (frexp), a bf16 value has 8
    significant bits, i.e. m is a multiple of 2**-8.  np.rint rounds half to
    even.  Only the normal range is handled (|x| >= 2**-126); smaller
    magnitudes are flushed to zero, larger than bf16's max overflow to inf.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    r = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    r = np.where(np.abs(x) < 2.0 ** -126, 0.0, r)
    big = 2.0 ** 127 * (2 - 2.0 ** -7)
    r = np.where(np.abs(r) > big, np.copysign(np.inf, r), r)
    return r


def round_f32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
