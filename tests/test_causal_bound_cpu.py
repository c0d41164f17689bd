"""Why causal attention is checked row by row.

Under the causal mask row i is a softmax over its own i + 1 keys.  With the
rounding points the kernel's storage types force (the weights P rounded to
bf16 before they multiply V, O stored in bf16; the row sum from the unrounded
weights), a row with a few keys carries errors of the order of 2^-9 |v|,
while the RMS of a slice that also holds rows with thousands of keys is of
the order of |v| / sqrt(#keys).  This test builds that exactly rounded
attention for a causal problem of 16,384 tokens, 2 heads, on rows 0..127 and
the last 896 rows, and checks the two facts the full-size causal GPU test
relies on: the slice-wide bound 2e-2 x RMS (+ 2^-8 |ref|) fails for such an
attention, and the same bound with each row's own RMS holds.
"""
import math

import numpy as np
import torch

import oracle as orc
from h3inputs import attention_qkv
from tests._parity import BF16_U, MAX_REL_RMS, MEAN_REL, assert_parity_rows


def _bf16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    return torch.from_numpy(a).to(torch.bfloat16).double().numpy()


def _causal_attention_rounded(qkv, H, rows, dh=128):
    """Causal softmax(q k^T / sqrt(dh)) v for the given query rows, the weights
    formed in fp32 and rounded to bf16 before they multiply v (the denominator
    keeps the unrounded fp32 weights), the result rounded to bf16."""
    L = qkv.shape[0]
    d = H * dh
    out = np.zeros((len(rows), d))
    for h in range(H):
        q = qkv[rows, h * dh:(h + 1) * dh]
        k = qkv[:, d + h * dh:d + (h + 1) * dh]
        v = qkv[:, 2 * d + h * dh:2 * d + (h + 1) * dh]
        s = (q @ k.T) / math.sqrt(dh)
        s = np.where(np.arange(L)[None, :] <= rows[:, None], s, -np.inf)
        p = np.exp(s - s.max(axis=1, keepdims=True)).astype(np.float32).astype(np.float64)
        out[:, h * dh:(h + 1) * dh] = _bf16((_bf16(p) @ v) / p.sum(axis=1, keepdims=True))
    return out


def test_causal_rows_need_their_own_rms():
    L, H = 16384, 2
    qkv = attention_qkv(L, H, seed=7).float().double().numpy()
    rows = np.concatenate([np.arange(128), np.arange(L - 896, L)]).astype(np.int64)
    ref, _ = orc.attention(qkv, H, 128, causal=True, rows=rows)
    got = _causal_attention_rounded(qkv, H, rows)
    rms = float(np.sqrt(np.mean(ref * ref)))
    slice_excess = float(np.max(np.abs(got - ref) - (MAX_REL_RMS * rms + BF16_U * np.abs(ref))))
    assert slice_excess > 0.0, slice_excess
    worst, mr = assert_parity_rows(got, ref, "exactly rounded causal attention")
    assert mr <= MEAN_REL
