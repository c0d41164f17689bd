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


def test_row_quantiser_definition():
    """Per row: scale = amax / 448, the largest magnitude lands on code +-448,
    every value within half a code step (times the scale) of its input, and an
    all-zero row keeps scale 1 and code 0."""
    from tests._fp8 import dequant_rows, quantize_rows

    rng = np.random.default_rng(3)
    x = (rng.normal(size=(6, 64)) * np.array([1e-3, 1, 7, 300, 1e4, 0])[:, None]).astype(np.float32)
    q, s = quantize_rows(x)
    amax = np.abs(x).max(axis=1)
    assert np.array_equal(s[:5], (amax[:5] / np.float32(448.0)).astype(np.float32))
    assert s[5] == 1.0 and np.all((q[5] & 0x7F) == 0)      # +0 or -0
    for r in range(5):
        i = int(np.argmax(np.abs(x[r])))
        assert (q[r, i] & 0x7F) == 0x7E and bool(q[r, i] & 0x80) == bool(x[r, i] < 0)
    deq = dequant_rows(x)
    t = np.abs(x / s[:, None].astype(np.float64))
    step = np.where(t < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(t, 2.0 ** -6))) - 3))
    assert np.all(np.abs(deq - x) <= 0.5 * step * s[:, None] * (1 + 1e-6))


def test_qk_quantiser_blocks():
    """Q: one scale per token and head; K: one scale per head and 128-key
    block (the ragged last block over its own keys only); V untouched."""
    from tests._fp8 import dequant_qk, dequant_rows

    rng = np.random.default_rng(4)
    L, H, dh = 300, 2, 128
    d = H * dh
    qkv = rng.normal(size=(L, 3 * d)).astype(np.float32)
    qkv[:, d:2 * d] *= np.repeat(np.array([1.0, 50.0, 0.01]), [128, 128, 44])[:, None]
    out = dequant_qk(qkv, H)
    assert np.array_equal(out[:, 2 * d:], qkv[:, 2 * d:].astype(np.float64))
    for h in range(H):
        cq = slice(h * dh, (h + 1) * dh)
        assert np.array_equal(out[:, cq], dequant_rows(qkv[:, cq]))
        k = qkv[:, d + h * dh:d + (h + 1) * dh]
        kd = out[:, d + h * dh:d + (h + 1) * dh]
        for b0, b1 in ((0, 128), (128, 256), (256, 300)):
            blk, dq = k[b0:b1], kd[b0:b1]
            amax = np.abs(blk).max()
            # the block's largest magnitude is represented exactly by code 448
            i = np.unravel_index(np.argmax(np.abs(blk)), blk.shape)
            assert dq[i] == float(np.sign(blk[i])) * 448.0 * float(np.float32(amax) / np.float32(448.0))
            # and every other value within half a code step at the block's scale
            assert np.max(np.abs(dq - blk)) <= amax / 448.0 * 16.0
