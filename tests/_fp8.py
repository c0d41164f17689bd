"""E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
largest finite 448) from its definition (test helper, no method arithmetic)."""
import numpy as np


def e4m3_decode(b: np.ndarray) -> np.ndarray:
    """Value of E4M3 bytes."""
    b = b.astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1 + m / 8.0) * 2.0 ** (e - 7))
    return sign * val


# the 127 non-negative finite values, ascending with their codes 0x00..0x7E
_POS = e4m3_decode(np.arange(127))


def e4m3_round(t: np.ndarray) -> np.ndarray:
    """E4M3 byte of each value: round to nearest, ties to the even code,
    saturating at +-448; the sign bit follows the input's sign."""
    a = np.minimum(np.abs(np.asarray(t, dtype=np.float64)), 448.0)
    hi = np.clip(np.searchsorted(_POS, a), 1, 126)
    lo = hi - 1
    d_lo, d_hi = a - _POS[lo], _POS[hi] - a
    code = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    return (code | (np.signbit(t).astype(np.int64) << 7)).astype(np.uint8)
