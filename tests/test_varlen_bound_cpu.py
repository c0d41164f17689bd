"""Why segment (cu_seqlens) attention is checked row by row.

With cu_seqlens each query row is a softmax over the keys of its own segment
("Joint Audio-Video Generation in Production", §3 Packed Sequences and
Modality Identity Preservation), and segment lengths range from one token to
the whole sequence.  A row of a two-token segment is a weighted mean of two
value rows, of the order of |v|; a row of a 500-token segment is of the order
of |v| / sqrt(#keys), and such rows set the RMS of the whole output.

A one-pass (online) softmax takes each row's weights against a reference
maximum and rounds them to bf16 before they multiply V.  The library's kernel
keeps the reference of the row's first visible key block until a later block
exceeds it by more than 8 in log2 units (a "lazy" rescale), so in a two-token
segment whose keys sit in consecutive blocks the larger weight, up to 2^8, is
the rounded one: an error of up to 2^-9 |v| on a row whose own magnitude can
be far below |v| (the two values cancel) and far above the slice RMS.

This test builds that arithmetic exactly (fp32 weights and row sums, bf16
weights into the numerator, O stored in bf16, key blocks of 128 from the
pair's first segment start as the kernel walks them) for the segments
[0, 511, 513, 1025, 1537] with 2 heads, and checks three facts: the slice-wide
bound 2e-2 x RMS (+ 2^-8 |ref|) fails for it, the same bound with each row's
own RMS holds, and with every weight taken against the row's true maximum (the
largest weight exactly 1) the slice-wide bound holds, so the lazy reference is
what the row-wise reading absorbs.
"""
import math

import numpy as np
import torch

import oracle as orc
from h3inputs import attention_qkv
from tests._parity import BF16_U, MAX_REL_RMS, MEAN_REL, assert_parity_rows, stats

CU = [0, 511, 513, 1025, 1537]
H = 2
SEED = CU[-1] + len(CU)          # the seed of the GPU segment-parity case
DH = 128
PAIR_ROWS = 512                  # query rows that share one walk over the keys
BLOCK = 128                      # keys per block
THRESHOLD = 8.0                  # log2 units


def _bf16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    return torch.from_numpy(a).to(torch.bfloat16).double().numpy()


def _segment_of(cu, L):
    cu = np.asarray(cu)
    seg = np.searchsorted(cu, np.arange(L), side="right") - 1
    return seg, cu[seg], cu[seg + 1]


def _online_lazy(qkv, cu, H, dh=DH):
    L = qkv.shape[0]
    d = H * dh
    c = math.log2(math.e) / math.sqrt(dh)
    seg, lo, hi = _segment_of(cu, L)
    out = np.zeros((L, d))
    for c0 in range(0, L, PAIR_ROWS):
        rows = np.arange(c0, min(c0 + PAIR_ROWS, L))
        kv_lo, kv_hi = cu[seg[rows[0]]], cu[seg[rows[-1]] + 1]
        for h in range(H):
            q = qkv[rows, h * dh:(h + 1) * dh]
            m = np.full(len(rows), -np.inf)
            l = np.zeros(len(rows), dtype=np.float32)
            o = np.zeros((len(rows), dh))
            for b0 in range(kv_lo, kv_hi, BLOCK):
                keys = np.arange(b0, min(b0 + BLOCK, L))
                k = qkv[keys, d + h * dh:d + (h + 1) * dh]
                v = qkv[keys, 2 * d + h * dh:2 * d + (h + 1) * dh]
                s = (q @ k.T).astype(np.float32).astype(np.float64)
                vis = (keys[None, :] >= lo[rows, None]) & (keys[None, :] < hi[rows, None])
                s = np.where(vis, s, -np.inf)
                mx = np.float32(c) * s.max(axis=1)
                need = mx > m + THRESHOLD
                with np.errstate(invalid="ignore"):
                    f = np.where(need, np.where(np.isinf(m), 0.0, np.exp2(m - mx)), 1.0)
                o *= f[:, None]
                l = (l * f).astype(np.float32)
                m = np.where(need, mx, m)
                ref = np.where(np.isinf(m), 0.0, m)
                p = np.exp2(np.float32(c) * s - ref[:, None]).astype(np.float32)
                l = (l + p.sum(axis=1, dtype=np.float32)).astype(np.float32)
                o += _bf16(p) @ v
            out[rows, h * dh:(h + 1) * dh] = _bf16(o / l[:, None].astype(np.float64))
    return out


def _true_max(qkv, cu, H, dh=DH):
    L = qkv.shape[0]
    d = H * dh
    out = np.zeros((L, d))
    for a, b in zip(cu[:-1], cu[1:]):
        for h in range(H):
            q = qkv[a:b, h * dh:(h + 1) * dh]
            k = qkv[a:b, d + h * dh:d + (h + 1) * dh]
            v = qkv[a:b, 2 * d + h * dh:2 * d + (h + 1) * dh]
            s = q @ k.T / math.sqrt(dh)
            p = np.exp(s - s.max(axis=1, keepdims=True)).astype(np.float32).astype(np.float64)
            out[a:b, h * dh:(h + 1) * dh] = _bf16((_bf16(p) @ v) / p.sum(axis=1, keepdims=True))
    return out


def _slice_excess(got, ref):
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(np.max(np.abs(got - ref) - (MAX_REL_RMS * rms + BF16_U * np.abs(ref))))


def test_segment_rows_need_their_own_rms():
    qkv = attention_qkv(CU[-1], H, seed=SEED).float().double().numpy()
    ref, _ = orc.attention_varlen(qkv, CU, H, DH)
    lazy = _online_lazy(qkv, CU, H)
    assert _slice_excess(lazy, ref) > 0.0
    worst, mr = assert_parity_rows(lazy, ref, "exactly rounded online softmax, lazy reference")
    assert mr <= MEAN_REL
    # the largest weight of each row exact: the slice-wide bound holds
    exact_max = _true_max(qkv, CU, H)
    assert _slice_excess(exact_max, ref) <= 0.0
    assert stats(exact_max, ref)[1] <= MEAN_REL


def test_lazy_emulation_is_the_oracle_without_rounding():
    """The emulation's walk (blocks, masks, lazy reference) without the two
    bf16 roundings reproduces the oracle to fp32 accuracy, so the failure
    above is the rounding alone."""
    global _bf16
    qkv = attention_qkv(700, 1, seed=3).float().double().numpy()
    cu = [0, 7, 7, 130, 300, 301, 700]
    ref, _ = orc.attention_varlen(qkv, cu, 1, DH)
    keep = _bf16
    try:
        _bf16 = lambda a: np.asarray(a, dtype=np.float64)  # noqa: E731
        got = _online_lazy(qkv, cu, 1)
    finally:
        _bf16 = keep
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-5 * float(np.abs(ref).max()))
