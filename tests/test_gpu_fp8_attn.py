"""Joint attention with E4M3 scores (the quantised-attention prior art that
"Joint Audio-Video Generation in Production", §6 names; Q and K in E4M3 with a
per-token Q scale and a per-128-key-block K scale, P V in bf16).

Three checks:
  - the quantiser's codes and scales, bit-exact against round-to-nearest-even
    E4M3 of x * (448 / amax) taken in fp32 (the precision the kernel decides
    them in), from the format's definition;
  - the kernel against the fp64 oracle run on Q and K quantised here in the
    test (that same definition, no value taken from the GPU): the block's
    bf16 tolerances, since the kernel computes exactly that attention up to
    the bf16 rounding of P and O;
  - the effect of the quantisation against the exact oracle, on rows that see
    at least 128 keys: mean relative error <= 0.08, the fp8 projections' bound
    (the bf16 error model with E4M3's unit roundoff 2^-4 in place of 2^-8,
    x16), and max |err| <= 0.64 RMS, twice their max bound: every score term
    carries two E4M3 roundings (of q and of k) and the softmax passes a score
    error to every weight of its row.  Rows with a handful of keys (the first
    causal rows, peaked rows) keep single score errors unaveraged and are
    covered by the second check only."""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from h3inputs import CONFIGS, attention_qkv
from tests._fp8 import codes_and_scale, dequant_qk, e4m3_decode
from tests._parity import assert_parity, slice_rows, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"
FP8_MAX, FP8_MEAN = 16 * 2e-2, 16 * 5e-3
SCORE_MAX = 2 * FP8_MAX


def _workspace(h3, L, H):
    n = h3.h3_attn_workspace_size_fp8(L, H)
    return torch.empty(n, dtype=torch.uint8, device=DEV), n


def _quantize(h3, qkv, L, H):
    d = H * 128
    nkb = (L + 127) // 128
    qk8 = torch.empty(L, 2 * d, dtype=torch.uint8, device=DEV)
    sq = torch.empty(H, L, dtype=torch.float32, device=DEV)
    sk = torch.empty(H, nkb, dtype=torch.float32, device=DEV)
    h3.h3_quantize_qk_fp8(qkv.to(DEV), L, H, 128, qk8, sq, sk)
    assert h3.h3_sync_status() == 0
    return qk8.cpu().numpy(), sq.cpu().numpy(), sk.cpu().numpy()


def _same_codes(got: np.ndarray, want: np.ndarray) -> bool:
    # +0 and -0 are the same value
    g = np.where((got & 0x7F) == 0, 0, got)
    w = np.where((want & 0x7F) == 0, 0, want)
    return np.array_equal(g, w)


@pytest.mark.parametrize("L,H", [(1, 1), (300, 2), (4096, 16)])
def test_quantize_qk_codes_and_scales_bit_exact(h3, L, H):
    qkv = attention_qkv(L, H, seed=70 + L, qk_std=1.5)
    d = H * 128
    if L >= 256:
        qkv[7, 0:128] = 0                      # an all-zero Q row of head 0
        qkv[128:256, d + 128:d + 256] = 0      # an all-zero K block of head 1
    qk8, sq, sk = _quantize(h3, qkv, L, H)
    x = qkv.float().numpy()
    nkb = (L + 127) // 128
    for h in range(H):
        q = x[:, h * 128:(h + 1) * 128]
        s_want, c_want = codes_and_scale(q, np.abs(q).max(axis=1, keepdims=True))
        assert np.array_equal(sq[h], s_want[:, 0]), f"Q scales, head {h}"
        assert _same_codes(qk8[:, h * 128:(h + 1) * 128], c_want), f"Q codes, head {h}"
        k = x[:, d + h * 128:d + (h + 1) * 128]
        for b in range(nkb):
            kb = k[b * 128:(b + 1) * 128]
            s_want, c_want = codes_and_scale(kb, np.abs(kb).max(keepdims=True))
            assert sk[h, b] == s_want.reshape(-1)[0], f"K scale, head {h} block {b}"
            got = qk8[b * 128:(b + 1) * 128, d + h * 128:d + (h + 1) * 128]
            assert _same_codes(got, c_want), f"K codes, head {h} block {b}"
    if L >= 256:
        assert sq[0, 7] == 1.0 and np.all(qk8[7, 0:128] & 0x7F == 0)
        assert sk[1, 1] == 1.0
    # every group's largest magnitude is the largest code
    assert np.abs(e4m3_decode(qk8[:, :128])).max() == 448.0


def _check(O, qkv, H, causal, what, lse=None, exact=True):
    oq, lq = orc.attention(dequant_qk(qkv.float().numpy(), H), H, 128, causal=bool(causal))
    assert_parity(to64(O), oq, what + " vs quantised-input oracle")
    if lse is not None:
        np.testing.assert_allclose(to64(lse), lq, atol=2e-2, rtol=1e-3)
    if exact:
        ro, _ = orc.attention(to64(qkv), H, 128, causal=bool(causal))
        rows = slice(127, None) if causal else slice(None)
        if ro[rows].size:
            assert_parity(to64(O)[rows], ro[rows], what + " vs exact oracle",
                          max_rel_rms=SCORE_MAX, mean_rel=FP8_MEAN)


@pytest.mark.parametrize("L,H,causal", [(1, 1, 0), (129, 2, 0), (257, 2, 1), (1000, 2, 0),
                                        (600, 2, 1), (4096, 4, 0), (513, 1, 0), (1025, 2, 1)])
def test_attention_fp8_parity(h3, L, H, causal):
    qkv = attention_qkv(L, H, seed=L + H + 7)
    ws, n = _workspace(h3, L, H)
    O = torch.full((L, H * 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((H, L), float("nan"), dtype=torch.float32, device=DEV)
    h3.h3_joint_attn_fwd_fp8(qkv.to(DEV), L, H, 128, causal, 1 / math.sqrt(128), ws, n, O, lse)
    assert h3.h3_sync_status() == 0
    _check(O, qkv, H, causal, f"fp8 attention L={L} H={H} causal={causal}", lse=lse)


@pytest.mark.parametrize("qk_std", [0.3, 2.0])
def test_attention_fp8_softmax_sharpness(h3, qk_std):
    """Flat to peaked rows; a peaked row has few effective keys, so only the
    quantised-input check applies to it."""
    L, H = 700, 1
    qkv = attention_qkv(L, H, seed=22, qk_std=qk_std)
    ws, n = _workspace(h3, L, H)
    O = torch.full((L, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    h3.h3_joint_attn_fwd_fp8(qkv.to(DEV), L, H, 128, 0, 1 / math.sqrt(128), ws, n, O)
    assert h3.h3_sync_status() == 0
    _check(O, qkv, H, 0, f"fp8 attention qk_std={qk_std}", exact=qk_std < 1)


def test_attention_fp8_identical_keys_give_mean_of_values(h3):
    """All keys equal: every score of a row is the same, so the softmax is flat
    whatever the rounding of Q and K."""
    L, H = 333, 1
    qkv = attention_qkv(L, H, seed=5)
    qkv[:, 128:256] = qkv[0:1, 128:256]
    ws, n = _workspace(h3, L, H)
    O = torch.empty(L, 128, dtype=torch.bfloat16, device=DEV)
    h3.h3_joint_attn_fwd_fp8(qkv.to(DEV), L, H, 128, 0, 1 / math.sqrt(128), ws, n, O)
    assert h3.h3_sync_status() == 0
    want = to64(qkv)[:, 256:].mean(axis=0)
    assert_parity(to64(O), np.tile(want, (L, 1)), "fp8 identical keys")


def test_attention_fp8_full_size_slice_rows(h3):
    c = CONFIGS["full"]
    L, H = c.L, c.n_heads
    qkv = attention_qkv(L, H, seed=59)
    ws, n = _workspace(h3, L, H)
    O = torch.full((L, H * 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    h3.h3_joint_attn_fwd_fp8(qkv.to(DEV), L, H, 128, 0, 1 / math.sqrt(128), ws, n, O)
    assert h3.h3_sync_status() == 0
    assert torch.isfinite(O.float()).all()
    rows = slice_rows(L, c.n_text)
    ridx = torch.from_numpy(rows).to(DEV)
    oq, _ = orc.attention(dequant_qk(qkv.float().numpy(), H), H, 128, rows=rows)
    assert_parity(to64(O[ridx]), oq, "fp8 full-size attention, slice rows, vs quantised-input oracle")
    ro, _ = orc.attention(to64(qkv), H, 128, rows=rows)
    assert_parity(to64(O[ridx]), ro, "fp8 full-size attention, slice rows, vs exact",
                  max_rel_rms=SCORE_MAX, mean_rel=FP8_MEAN)
