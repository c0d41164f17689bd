"""The E4M3 helper the fp8 GPU tests compare against, pinned to the format's
definition: every finite code round-trips, midpoints go to the even code,
values past 448 saturate, and the spacing is 2^(e-3) (2^-9 below 2^-6)."""
import numpy as np

from tests._fp8 import e4m3_decode, e4m3_round


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = e4m3_decode(codes)
    back = e4m3_round(np.where(codes & 0x80, -1.0, 1.0) * np.abs(vals))
    assert np.array_equal(back, codes)


def test_known_values_and_spacing():
    assert e4m3_decode(np.array([0x38]))[0] == 1.0           # exponent field 7 = bias
    assert e4m3_decode(np.array([0x7E]))[0] == 448.0         # largest finite
    assert e4m3_decode(np.array([0x01]))[0] == 2.0 ** -9     # smallest subnormal
    assert e4m3_decode(np.array([0x08]))[0] == 2.0 ** -6     # smallest normal
    pos = e4m3_decode(np.arange(127))
    assert np.all(np.diff(pos) > 0)
    for e in range(1, 16):
        block = pos[e * 8:e * 8 + 8] if e < 15 else pos[120:127]
        assert np.allclose(np.diff(block), 2.0 ** (e - 7 - 3))


def test_rounding_to_nearest_even_and_saturation():
    pos = e4m3_decode(np.arange(127))
    mid = (pos[:-1] + pos[1:]) / 2
    got = e4m3_round(mid)
    lo = np.arange(126)
    want = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(got, want.astype(np.uint8))
    assert np.array_equal(e4m3_round(mid - 1e-12), lo.astype(np.uint8))
    assert np.array_equal(e4m3_round(mid + 1e-12), (lo + 1).astype(np.uint8))
    assert e4m3_round(np.array([1e6]))[0] == 0x7E and e4m3_round(np.array([-1e6]))[0] == 0xFE
