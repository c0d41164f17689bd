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


_F448 = np.float32(448.0)


def codes_and_scale(x32: np.ndarray, amax: np.ndarray):
    """E4M3 codes of float32 values ``x32`` that share the maxima ``amax``
    (broadcast against x32), and the group scales amax / 448 (1 for an
    all-zero group).  Both decisions are taken in float32, the precision the
    quantising kernels take them in: x * (448 / amax) rounded to the nearest
    code, ties to even, saturating."""
    x32 = np.asarray(x32, dtype=np.float32)
    amax = np.asarray(amax, dtype=np.float32)
    nz = amax > 0
    scale = np.where(nz, amax / _F448, np.float32(1.0)).astype(np.float32)
    inv = np.where(nz, _F448 / np.where(nz, amax, np.float32(1.0)),
                   np.float32(1.0)).astype(np.float32)
    return scale, e4m3_round((x32 * inv).astype(np.float32))


def quantize_rows(x: np.ndarray):
    """Row-wise quantisation of ``x [R, K]``: (codes [R, K], scales [R])."""
    x32 = np.asarray(x, dtype=np.float32)
    s, q = codes_and_scale(x32, np.abs(x32).max(axis=1, keepdims=True))
    return q, s[:, 0]


def dequant_rows(x: np.ndarray) -> np.ndarray:
    """The float64 values a row-quantised operand stands for: code x scale."""
    q, s = quantize_rows(x)
    return e4m3_decode(q) * s.astype(np.float64)[:, None]


def dequant_qk(qkv: np.ndarray, n_heads: int, head_dim: int = 128, block: int = 128
               ) -> np.ndarray:
    """``qkv [L, 3*H*dh]`` with Q replaced by its per-token E4M3 values and K by
    its per-(head, 128-key block) E4M3 values, times their scales; V as is."""
    x = np.asarray(qkv, dtype=np.float32)
    L, d = x.shape[0], n_heads * head_dim
    nb = (L + block - 1) // block
    out = np.asarray(qkv, dtype=np.float64).copy()
    for h in range(n_heads):
        cq = slice(h * head_dim, (h + 1) * head_dim)
        out[:, cq] = dequant_rows(x[:, cq])
        # K blocks of 128 keys (the last one padded with zeros, which change no maximum)
        k = np.zeros((nb * block, head_dim), dtype=np.float32)
        k[:L] = x[:, d + h * head_dim:d + (h + 1) * head_dim]
        kb = k.reshape(nb, block * head_dim)
        s, q = codes_and_scale(kb, np.abs(kb).max(axis=1, keepdims=True))
        deq = e4m3_decode(q) * s.astype(np.float64)
        out[:, d + h * head_dim:d + (h + 1) * head_dim] = deq.reshape(nb * block, head_dim)[:L]
    return out
