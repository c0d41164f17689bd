"""The FP8 (E4M3) variant of the projections ("Joint Audio-Video Generation
in Production", §5: the active block held at FP8 - prior art).  The oracle is
the same fp64 computation on the bf16 inputs; the tolerance follows the bf16
bounds' error model with the E4M3 unit roundoff 2^-4 in place of bf16's 2^-8:
both bounds scaled by 16 (max |err| <= 0.32 RMS, mean relative <= 0.08)."""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from h3inputs import CONFIGS, block_inputs
from tests._fp8 import e4m3_decode
from tests._parity import assert_parity, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"
FP8_MAX, FP8_MEAN = 16 * 2e-2, 16 * 5e-3


def _quant(h3, x):
    R, K = x.shape
    q = torch.empty(R, K, dtype=torch.uint8, device=DEV)
    s = torch.empty(R, dtype=torch.float32, device=DEV)
    h3.h3_quantize_rows_fp8(x, R, K, q, s)
    return q, s


def test_quantize_rows_grid_and_maximum(h3):
    g = torch.Generator().manual_seed(40)
    x = (torch.randn(300, 5120, generator=g) * torch.rand(300, 1, generator=g) * 5)
    x[7] = 0.0                                          # an all-zero row
    xb = x.to(torch.bfloat16)
    q, s = _quant(h3, xb.to(DEV))
    assert h3.h3_sync_status() == 0
    qv = e4m3_decode(q.cpu().numpy())
    sv = s.cpu().double().numpy()
    xv = to64(xb)
    assert sv[7] == 1.0 and np.all(qv[7] == 0)
    # the largest element of every row maps to +-448
    amax = np.abs(xv).max(axis=1)
    nz = amax > 0
    np.testing.assert_allclose(sv[nz], amax[nz] / 448.0, rtol=1e-6)
    big = np.abs(qv[nz]).max(axis=1)
    assert np.all(big == 448.0)
    # every value within half an E4M3 spacing of x / s (3 mantissa bits; subnormal
    # spacing 2^-9)
    t = xv / sv[:, None]
    assert np.all(np.abs(qv - t) <= np.maximum(np.abs(t) * 2.0 ** -4, 2.0 ** -10) + 1e-9)


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (300, 384, 512), (1000, 2048, 2048)])
def test_gemm_fp8_against_oracle(h3, M, N, K):
    g = torch.Generator().manual_seed(M + N + K)
    a = torch.randn(M, K, generator=g).to(torch.bfloat16)
    b = (torch.randn(N, K, generator=g) / math.sqrt(K)).to(torch.bfloat16)
    qa, sa = _quant(h3, a.to(DEV))
    qb, sb = _quant(h3, b.to(DEV))
    c = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    h3.h3_gemm_fp8(qa, sa, qb, sb, M, N, K, c)
    assert h3.h3_sync_status() == 0
    assert_parity(to64(c), orc.linear(to64(a), to64(b)), f"gemm fp8 {M}x{N}x{K}",
                  max_rel_rms=FP8_MAX, mean_rel=FP8_MEAN)


def _quantized_weights(h3, *ws):
    out = []
    for w in ws:
        q, s = _quant(h3, w.to(DEV))
        out += [q, s]
    return out


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_block_fp8_against_oracle(h3, name):
    c = CONFIGS[name]
    inp = block_inputs(c)
    args = (c.n_text, c.video_t, c.video_h, c.video_w, c.audio_channels, c.audio_steps)
    mod, pos = h3.h3_build_packed_layout(*args)
    omod, opos = orc.packed_layout(*args)
    desc = h3.BlockDesc.make(L=c.L, d=c.d, n_heads=c.n_heads)
    nbytes = h3.h3_workspace_size_fp8(desc)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    out = torch.full((c.L, c.d), float("nan"), dtype=torch.bfloat16, device=DEV)
    dv = {k: v.to(DEV) for k, v in inp.items() if k != "x_raw"}
    wq, wqs, woq, wos = _quantized_weights(h3, inp["Wqkv"], inp["Wo"])
    h3.h3_attn_block_fwd_fp8(desc, dv["x"], torch.from_numpy(mod).to(DEV),
                             torch.from_numpy(pos).to(DEV), dv["shift"], dv["scale"], dv["gate"],
                             wq, wqs, woq, wos, ws, nbytes, out)
    assert h3.h3_sync_status() == 0
    f = lambda k: to64(inp[k])
    r = orc.block(f("x"), omod, opos, f("shift"), f("scale"), f("gate"), f("Wqkv"), f("Wo"),
                  c.n_heads)
    off = (c.L * c.d * 2 + 255) // 256 * 256
    qkv = ws[off:off + c.L * 3 * c.d * 2].view(torch.bfloat16).view(c.L, 3 * c.d)
    assert_parity(to64(qkv), r["qkv"], f"{name} fp8 qkv", max_rel_rms=FP8_MAX, mean_rel=FP8_MEAN)
    assert_parity(to64(out), r["out"], f"{name} fp8 out", max_rel_rms=FP8_MAX,
                  mean_rel=FP8_MEAN, bf16_storage=False)


def test_mlp_fp8_against_oracle(h3):
    c = CONFIGS["small"]
    hidden = 4 * c.d
    g = torch.Generator().manual_seed(41)
    x = torch.randn(c.L, c.d, generator=g).to(torch.bfloat16)
    w1 = (torch.randn(hidden, c.d, generator=g) / math.sqrt(c.d)).to(torch.bfloat16)
    w2 = (torch.randn(c.d, hidden, generator=g) / math.sqrt(hidden)).to(torch.bfloat16)
    sh, sc, gt = (torch.randn(3, c.d, generator=g) * 0.1 for _ in range(3))
    mod, _ = h3.h3_build_packed_layout(c.n_text, c.video_t, c.video_h, c.video_w,
                                       c.audio_channels, c.audio_steps)
    desc = h3.MlpDesc.make(L=c.L, d=c.d, hidden=hidden)
    nbytes = h3.h3_mlp_workspace_size_fp8(desc)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    out = torch.empty(c.L, c.d, dtype=torch.bfloat16, device=DEV)
    w1q, w1s, w2q, w2s = _quantized_weights(h3, w1, w2)
    h3.h3_mlp_block_fwd_fp8(desc, x.to(DEV), torch.from_numpy(mod).to(DEV), sh.to(DEV), sc.to(DEV),
                            gt.to(DEV), w1q, w1s, w2q, w2s, ws, nbytes, out)
    assert h3.h3_sync_status() == 0
    r = orc.mlp_block(to64(x), mod, to64(sh), to64(sc), to64(gt), to64(w1), to64(w2))
    assert_parity(to64(out), r["out"], "small fp8 mlp out", max_rel_rms=FP8_MAX,
                  mean_rel=FP8_MEAN, bf16_storage=False)


def test_block_fp8_with_segments_against_oracle(h3):
    """With cu_seqlens the fp8 block keeps its fp8 projections and attends per
    segment in bf16 (the fp8 scores are for the unsegmented sequence only)."""
    c = CONFIGS["small"]
    cu = [0, c.n_text, c.n_text + c.n_video, c.L]
    inp = block_inputs(c)
    args = (c.n_text, c.video_t, c.video_h, c.video_w, c.audio_channels, c.audio_steps)
    mod, pos = h3.h3_build_packed_layout(*args)
    omod, opos = orc.packed_layout(*args)
    desc = h3.BlockDesc.make(L=c.L, d=c.d, n_heads=c.n_heads, cu_seqlens=cu)
    nbytes = h3.h3_workspace_size_fp8(desc)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    out = torch.full((c.L, c.d), float("nan"), dtype=torch.bfloat16, device=DEV)
    dv = {k: v.to(DEV) for k, v in inp.items() if k != "x_raw"}
    wq, wqs, woq, wos = _quantized_weights(h3, inp["Wqkv"], inp["Wo"])
    h3.h3_attn_block_fwd_fp8(desc, dv["x"], torch.from_numpy(mod).to(DEV),
                             torch.from_numpy(pos).to(DEV), dv["shift"], dv["scale"], dv["gate"],
                             wq, wqs, woq, wos, ws, nbytes, out)
    assert h3.h3_sync_status() == 0
    f = lambda k: to64(inp[k])
    r = orc.block(f("x"), omod, opos, f("shift"), f("scale"), f("gate"), f("Wqkv"), f("Wo"),
                  c.n_heads, cu_seqlens=cu)
    assert_parity(to64(out), r["out"], "small fp8 block with segments", max_rel_rms=FP8_MAX,
                  mean_rel=FP8_MEAN, bf16_storage=False)
