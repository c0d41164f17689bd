"""The FP8 (E4M3) variant of the projections ("Joint Audio-Video Generation
in Production", §5: the active block held at FP8 - prior art).

Two checks per call:
  - against the fp64 oracle fed the E4M3 operands that the call's definition
    implies, quantised here in the test from the format's definition (per-row
    scale amax / 448 for activations and for weight output channels,
    round-to-nearest-even, decided in fp32 on the bf16 values the fp8 path
    stores, as the kernels decide them; no value is taken from the GPU): the
    bf16 bounds of the block, because the kernels compute exactly that product
    up to their bf16 storage;
  - the effect of the quantisation against the exact oracle: the bf16 bounds'
    error model with the E4M3 unit roundoff 2^-4 in place of bf16's 2^-8, both
    bounds scaled by 16 (max |err| <= 0.32 RMS, mean relative <= 0.08).
The row quantiser itself is compared bit for bit with that definition."""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from h3inputs import CONFIGS, block_inputs
from tests._fp8 import dequant_qk, dequant_rows, e4m3_decode, quantize_rows
from tests._parity import CHAIN_MAX_REL_RMS, assert_parity, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"
FP8_MAX, FP8_MEAN = 16 * 2e-2, 16 * 5e-3


def _quant(h3, x):
    R, K = x.shape
    q = torch.empty(R, K, dtype=torch.uint8, device=DEV)
    s = torch.empty(R, dtype=torch.float32, device=DEV)
    h3.h3_quantize_rows_fp8(x, R, K, q, s)
    return q, s


def _same_codes(got: np.ndarray, want: np.ndarray) -> bool:
    # +0 and -0 are the same value
    g = np.where((got & 0x7F) == 0, 0, got)
    w = np.where((want & 0x7F) == 0, 0, want)
    return np.array_equal(g, w)


def test_quantize_rows_bit_exact(h3):
    g = torch.Generator().manual_seed(40)
    x = (torch.randn(300, 5120, generator=g) * torch.rand(300, 1, generator=g) * 5)
    x[7] = 0.0                                          # an all-zero row
    x[9] = 0.0
    x[9, 100] = 1e-30                                   # a row with one tiny value
    xb = x.to(torch.bfloat16)
    q, s = _quant(h3, xb.to(DEV))
    assert h3.h3_sync_status() == 0
    want_q, want_s = quantize_rows(xb.float().numpy())
    assert np.array_equal(s.cpu().numpy(), want_s)
    assert _same_codes(q.cpu().numpy(), want_q)
    qv = e4m3_decode(q.cpu().numpy())
    assert s[7].item() == 1.0 and np.all(qv[7] == 0)
    assert np.all(np.abs(qv[np.abs(to64(xb)).max(axis=1) > 0]).max(axis=1) == 448.0)


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (300, 384, 512), (1000, 2048, 2048),
                                   (1, 256, 256), (257, 512, 512)])
def test_gemm_fp8_against_oracle(h3, M, N, K):
    g = torch.Generator().manual_seed(M + N + K)
    a = torch.randn(M, K, generator=g).to(torch.bfloat16)
    b = (torch.randn(N, K, generator=g) / math.sqrt(K)).to(torch.bfloat16)
    qa, sa = _quant(h3, a.to(DEV))
    qb, sb = _quant(h3, b.to(DEV))
    c = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    h3.h3_gemm_fp8(qa, sa, qb, sb, M, N, K, c)
    assert h3.h3_sync_status() == 0
    a32, b32 = a.float().numpy(), b.float().numpy()
    assert_parity(to64(c), orc.linear(dequant_rows(a32), dequant_rows(b32)),
                  f"gemm fp8 {M}x{N}x{K} vs quantised-operand oracle")
    assert_parity(to64(c), orc.linear(to64(a), to64(b)), f"gemm fp8 {M}x{N}x{K} vs exact",
                  max_rel_rms=FP8_MAX, mean_rel=FP8_MEAN)


def _quantized_weights(h3, *ws):
    out = []
    for w in ws:
        q, s = _quant(h3, w.to(DEV))
        out += [q, s]
    return out


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).double().numpy()


def _fp8_block_oracle(o, mod, pos, H, cu=None):
    """The block with every E4M3 operand of the fp8 path quantised from its
    definition: y and O per token, Wqkv and Wo per output channel, and (without
    segments) Q per token and K per 128-key block for the scores.  The fp8 path
    quantises the bf16 values it stores (y, the rotated qkv, O), so each
    quantisation here decides its codes on the same bf16 values of the fp64
    chain; every product is then exact."""
    y = _bf16(orc.adaln_modulate(o["x"], mod, o["shift"], o["scale"]))
    qkv = orc.mrope(orc.linear(dequant_rows(y), dequant_rows(o["Wqkv"])), pos, H)
    if cu is None:
        O, _ = orc.attention(dequant_qk(_bf16(qkv), H), H)
    else:
        O, _ = orc.attention_varlen(qkv, cu, H)
    branch = orc.linear(dequant_rows(_bf16(O)), dequant_rows(o["Wo"]))
    return {"qkv": qkv, "O": O, "out": orc.gated_residual(o["x"], branch, mod, o["gate"])}


def _run_fp8_block(h3, c, inp, mod, pos, cu=None):
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
    off = (c.L * c.d * 2 + 255) // 256 * 256
    qkv = ws[off:off + c.L * 3 * c.d * 2].view(torch.bfloat16).view(c.L, 3 * c.d)
    O = ws[:c.L * c.d * 2].view(torch.bfloat16).view(c.L, c.d)
    return out, qkv, O


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_block_fp8_against_oracle(h3, name):
    c = CONFIGS[name]
    inp = block_inputs(c)
    args = (c.n_text, c.video_t, c.video_h, c.video_w, c.audio_channels, c.audio_steps)
    mod, pos = h3.h3_build_packed_layout(*args)
    omod, opos = orc.packed_layout(*args)
    out, qkv, O = _run_fp8_block(h3, c, inp, mod, pos)
    o = {k: to64(v) for k, v in inp.items() if k != "x_raw"}
    rq = _fp8_block_oracle(o, omod, opos, c.n_heads)
    assert_parity(to64(qkv), rq["qkv"], f"{name} fp8 qkv vs quantised-operand oracle")
    assert_parity(to64(O), rq["O"], f"{name} fp8 O vs quantised-operand oracle",
                  max_rel_rms=CHAIN_MAX_REL_RMS)
    assert_parity(to64(out), rq["out"], f"{name} fp8 out vs quantised-operand oracle",
                  bf16_storage=False)
    r = orc.block(o["x"], omod, opos, o["shift"], o["scale"], o["gate"], o["Wqkv"], o["Wo"],
                  c.n_heads)
    assert_parity(to64(qkv), r["qkv"], f"{name} fp8 qkv vs exact", max_rel_rms=FP8_MAX,
                  mean_rel=FP8_MEAN)
    assert_parity(to64(out), r["out"], f"{name} fp8 out vs exact", max_rel_rms=FP8_MAX,
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
    off = (c.L * c.d * 2 + 255) // 256 * 256
    h_gpu = ws[off:off + c.L * hidden * 2].view(torch.bfloat16).view(c.L, hidden)
    # the quantised-operand oracle: y and h per token (codes decided on their
    # bf16 values, as stored by the fp8 path), W1 and W2 per output channel
    x64, s64, c64, g64 = to64(x), to64(sh), to64(sc), to64(gt)
    y = _bf16(orc.adaln_modulate(x64, mod, s64, c64))
    h = orc.gelu_tanh(orc.linear(dequant_rows(y), dequant_rows(to64(w1))))
    branch = orc.linear(dequant_rows(_bf16(h)), dequant_rows(to64(w2)))
    assert_parity(to64(h_gpu), h, "small fp8 mlp h vs quantised-operand oracle")
    assert_parity(to64(out), orc.gated_residual(x64, branch, mod, g64),
                  "small fp8 mlp out vs quantised-operand oracle", bf16_storage=False)
    r = orc.mlp_block(x64, mod, s64, c64, g64, to64(w1), to64(w2))
    assert_parity(to64(out), r["out"], "small fp8 mlp out vs exact", max_rel_rms=FP8_MAX,
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
    out, qkv, O = _run_fp8_block(h3, c, inp, mod, pos, cu=cu)
    o = {k: to64(v) for k, v in inp.items() if k != "x_raw"}
    rq = _fp8_block_oracle(o, omod, opos, c.n_heads, cu=cu)
    assert_parity(to64(qkv), rq["qkv"], "fp8 block with segments: qkv vs quantised-operand oracle")
    assert_parity(to64(out), rq["out"], "fp8 block with segments: out vs quantised-operand oracle",
                  bf16_storage=False)
    r = orc.block(o["x"], omod, opos, o["shift"], o["scale"], o["gate"], o["Wqkv"], o["Wo"],
                  c.n_heads, cu_seqlens=cu)
    assert_parity(to64(out), r["out"], "fp8 block with segments: out vs exact",
                  max_rel_rms=FP8_MAX, mean_rel=FP8_MEAN, bf16_storage=False)


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_block_fp8_scores_equal_the_quantiser(h3, name):
    """Without segments the fp8 block's attention takes E4M3 Q and K (Q8 | K8
    and their scales, in the block's workspace); they equal, bit for bit, what
    h3_quantize_qk_fp8 forms from the rotated bf16 qkv the block left in its
    workspace."""
    c = CONFIGS[name]
    L, d, H = c.L, c.d, c.n_heads
    inp = block_inputs(c)
    args = (c.n_text, c.video_t, c.video_h, c.video_w, c.audio_channels, c.audio_steps)
    mod, pos = h3.h3_build_packed_layout(*args)
    desc = h3.BlockDesc.make(L=L, d=d, n_heads=H)
    nbytes = h3.h3_workspace_size_fp8(desc)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    out = torch.empty(L, d, dtype=torch.bfloat16, device=DEV)
    dv = {k: v.to(DEV) for k, v in inp.items() if k != "x_raw"}
    wq, wqs, woq, wos = _quantized_weights(h3, inp["Wqkv"], inp["Wo"])
    h3.h3_attn_block_fwd_fp8(desc, dv["x"], torch.from_numpy(mod).to(DEV),
                             torch.from_numpy(pos).to(DEV), dv["shift"], dv["scale"], dv["gate"],
                             wq, wqs, woq, wos, ws, nbytes, out)
    assert h3.h3_sync_status() == 0
    r256 = lambda n: (n + 255) // 256 * 256
    off_qkv = r256(L * d * 2)
    off_qk8 = off_qkv + r256(L * 3 * d * 2) + r256(L * d) + r256(L * 4)
    off_sq = off_qk8 + r256(L * 2 * d)
    off_sk = off_sq + r256(H * L * 4)
    nkb = (L + 127) // 128
    qkv = ws[off_qkv:off_qkv + L * 3 * d * 2].view(torch.bfloat16).view(L, 3 * d)
    qk8 = ws[off_qk8:off_qk8 + L * 2 * d]
    sq = ws[off_sq:off_sq + H * L * 4].view(torch.float32)
    sk = ws[off_sk:off_sk + H * nkb * 4].view(torch.float32)
    ref8 = torch.empty_like(qk8)
    rsq = torch.empty_like(sq)
    rsk = torch.empty_like(sk)
    h3.h3_quantize_qk_fp8(qkv, L, H, 128, ref8, rsq, rsk)
    assert h3.h3_sync_status() == 0
    assert torch.equal(qk8, ref8)
    assert torch.equal(sq.view(torch.int32), rsq.view(torch.int32))
    assert torch.equal(sk.view(torch.int32), rsk.view(torch.int32))
