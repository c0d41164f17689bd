"""A packed sequence longer than the full-size one: L = 150,000 tokens (358
text + 32 x 45 x 100 video + 2 x 2,821 audio), d = 5120, 40 heads.  The
fused block's qkv then holds 2.3e9 elements (its byte offsets pass 2^31
inside row 69,905 and 2^32 inside row 139,810, where its element offsets pass
2^31 too), so every row and pointer offset of the path has to be 64-bit.

Each stage is checked on sampled rows against the oracle, fed the stage's
input as the GPU consumed it ("Joint Audio-Video Generation in Production",
§1 Unified Architecture: one attention context over the whole packed
sequence; §6: exactly the L effective tokens take part): the rotated q, k, v
of the rows from x, attention of the rows over all 150,000 keys (heads 0 and
39) from the block's own qkv, and out of the rows from its own O."""
import numpy as np
import pytest
import torch

import oracle as orc
from h3inputs import BlockConfig, block_inputs_device, random_rows
from tests._parity import CHAIN_MAX_REL_RMS, assert_parity, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _rows(L: int, d: int) -> np.ndarray:
    n3 = 3 * d
    around = []
    for edge in (2 ** 31 // (2 * n3), 2 ** 32 // (2 * n3), 2 ** 31 // n3):
        around += [edge - 1, edge, edge + 1]
    rows = np.concatenate([np.arange(4), np.array(around), random_rows(L, 40, seed=31).numpy(),
                           np.arange(L - 8, L)])
    return np.unique(rows).astype(np.int64)


def test_long_sequence_block_sampled_rows(h3):
    c = BlockConfig("long", 358, 32, 45, 100, 2, 2821, d=5120, n_heads=40, seed=23)
    L, d, H = c.L, c.d, c.n_heads
    assert L == 150_000 and L * 3 * d > 2 ** 31
    inp = block_inputs_device(c, DEV)
    args = (c.n_text, c.video_t, c.video_h, c.video_w, c.audio_channels, c.audio_steps)
    mod, pos = h3.h3_build_packed_layout(*args)
    omod, opos = orc.packed_layout(*args)
    desc = h3.BlockDesc.make(L=L, d=d, n_heads=H)
    nbytes = h3.h3_workspace_size(desc)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    out = torch.full((L, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    dv = inp
    h3.h3_attn_block_fwd(desc, dv["x"], torch.from_numpy(mod).to(DEV),
                         torch.from_numpy(pos).to(DEV), dv["shift"], dv["scale"], dv["gate"],
                         dv["Wqkv"], dv["Wo"], ws, nbytes, out)
    assert h3.h3_sync_status() == 0
    off = (L * d * 2 + 255) // 256 * 256
    O = ws[:L * d * 2].view(torch.bfloat16).view(L, d)
    qkv = ws[off:off + L * 3 * d * 2].view(torch.bfloat16).view(L, 3 * d)
    assert torch.isfinite(out.float()).all()

    rows = _rows(L, d)
    ridx = torch.from_numpy(rows).to(DEV)
    m64 = {k: to64(inp[k]) for k in ("shift", "scale", "gate")}
    x_rows = to64(inp["x"][ridx])
    # q, k, v of the rows from x: modulate, projection, 3D RoPE
    y = orc.adaln_modulate(x_rows, omod[rows], m64["shift"], m64["scale"])
    ref_qkv = orc.mrope(orc.linear(y, to64(inp["Wqkv"])), opos[rows], H)
    got_qkv = to64(qkv[ridx])
    for b, name in enumerate("qkv"):
        assert_parity(got_qkv[:, b * d:(b + 1) * d], ref_qkv[:, b * d:(b + 1) * d],
                      f"L = {L}: {name} of the sampled rows")
    # attention of the rows over all keys, from the block's own qkv (heads 0 and 39)
    heads = (0, H - 1)
    cols = np.concatenate([np.arange(blk * d + h * 128, blk * d + (h + 1) * 128)
                           for blk in range(3) for h in heads])
    sub = to64(qkv[:, torch.from_numpy(cols).to(DEV)])
    ref_o, _ = orc.attention(sub, len(heads), 128, rows=rows)
    ocols = torch.from_numpy(np.concatenate([np.arange(h * 128, (h + 1) * 128)
                                             for h in heads])).to(DEV)
    assert_parity(to64(O[ridx][:, ocols]), ref_o, f"L = {L}: O of the sampled rows, heads {heads}",
                  max_rel_rms=CHAIN_MAX_REL_RMS)
    # out of the rows from the block's own O
    ref_out = orc.gated_residual(x_rows, orc.linear(to64(O[ridx]), to64(inp["Wo"])), omod[rows],
                                 m64["gate"])
    assert_parity(to64(out[ridx]), ref_out, f"L = {L}: out of the sampled rows", bf16_storage=False)
    del ws, out, dv, inp, qkv, O
    torch.cuda.empty_cache()


def test_long_sequence_fp8_block_sampled_rows(h3):
    """The fp8 block at the same length, stage by stage against the
    quantised-operand oracle (E4M3 codes decided in the test from the format's
    definition on the bf16 values the fp8 path stores; see test_gpu_fp8.py)."""
    from tests._fp8 import dequant_qk, dequant_rows
    from tests.test_gpu_fp8 import _bf16, _quantized_weights

    c = BlockConfig("long", 358, 32, 45, 100, 2, 2821, d=5120, n_heads=40, seed=23)
    L, d, H = c.L, c.d, c.n_heads
    inp = block_inputs_device(c, DEV)
    args = (c.n_text, c.video_t, c.video_h, c.video_w, c.audio_channels, c.audio_steps)
    mod, pos = h3.h3_build_packed_layout(*args)
    omod, opos = orc.packed_layout(*args)
    desc = h3.BlockDesc.make(L=L, d=d, n_heads=H)
    nbytes = h3.h3_workspace_size_fp8(desc)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    out = torch.full((L, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    wq, wqs, woq, wos = _quantized_weights(h3, inp["Wqkv"], inp["Wo"])
    h3.h3_attn_block_fwd_fp8(desc, inp["x"], torch.from_numpy(mod).to(DEV),
                             torch.from_numpy(pos).to(DEV), inp["shift"], inp["scale"],
                             inp["gate"], wq, wqs, woq, wos, ws, nbytes, out)
    assert h3.h3_sync_status() == 0
    off = (L * d * 2 + 255) // 256 * 256
    O = ws[:L * d * 2].view(torch.bfloat16).view(L, d)
    qkv = ws[off:off + L * 3 * d * 2].view(torch.bfloat16).view(L, 3 * d)

    rows = _rows(L, d)
    ridx = torch.from_numpy(rows).to(DEV)
    m64 = {k: to64(inp[k]) for k in ("shift", "scale", "gate")}
    x_rows = to64(inp["x"][ridx])
    y = _bf16(orc.adaln_modulate(x_rows, omod[rows], m64["shift"], m64["scale"]))
    ref_qkv = orc.mrope(orc.linear(dequant_rows(y), dequant_rows(to64(inp["Wqkv"]))), opos[rows], H)
    assert_parity(to64(qkv[ridx]), ref_qkv, f"fp8 block, L = {L}: qkv of the sampled rows")
    heads = (0, H - 1)
    cols = np.concatenate([np.arange(blk * d + h * 128, blk * d + (h + 1) * 128)
                           for blk in range(3) for h in heads])
    sub = to64(qkv[:, torch.from_numpy(cols).to(DEV)])
    ref_o, _ = orc.attention(dequant_qk(sub, len(heads)), len(heads), 128, rows=rows)
    ocols = torch.from_numpy(np.concatenate([np.arange(h * 128, (h + 1) * 128)
                                             for h in heads])).to(DEV)
    assert_parity(to64(O[ridx][:, ocols]), ref_o,
                  f"fp8 block, L = {L}: O of the sampled rows, heads {heads}",
                  max_rel_rms=CHAIN_MAX_REL_RMS)
    branch = orc.linear(dequant_rows(to64(O[ridx])), dequant_rows(to64(inp["Wo"])))
    assert_parity(to64(out[ridx]), orc.gated_residual(x_rows, branch, omod[rows], m64["gate"]),
                  f"fp8 block, L = {L}: out of the sampled rows", bf16_storage=False)
    del ws, out, inp, qkv, O, wq, wqs, woq, wos
    torch.cuda.empty_cache()


def test_long_sequence_mlp_sampled_rows(h3):
    """The MLP sub-block (hidden 4d) at L = 150,000: its GELU output h holds
    3.07e9 elements (byte offsets past 2^31 inside row 52,428 and past 2^32
    inside row 104,857, where the element offsets pass 2^31)."""
    c = BlockConfig("long", 358, 32, 45, 100, 2, 2821, d=5120, n_heads=40, seed=23)
    L, d = c.L, c.d
    hidden = 4 * d
    x = block_inputs_device(c, DEV)["x"]
    g = torch.Generator(device=DEV)
    g.manual_seed(29)
    w1 = (torch.randn(hidden, d, generator=g, device=DEV) / d ** 0.5).to(torch.bfloat16)
    w2 = (torch.randn(d, hidden, generator=g, device=DEV) / hidden ** 0.5).to(torch.bfloat16)
    sh, sc, gt = (torch.randn(3, d, generator=g, device=DEV) * 0.1 for _ in range(3))
    mod, _ = h3.h3_build_packed_layout(c.n_text, c.video_t, c.video_h, c.video_w,
                                       c.audio_channels, c.audio_steps)
    desc = h3.MlpDesc.make(L=L, d=d, hidden=hidden)
    nbytes = h3.h3_mlp_workspace_size(desc)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    out = torch.full((L, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    h3.h3_mlp_block_fwd(desc, x, torch.from_numpy(mod).to(DEV), sh, sc, gt, w1, w2, ws, nbytes,
                        out)
    assert h3.h3_sync_status() == 0
    off = (L * d * 2 + 255) // 256 * 256
    h = ws[off:off + L * hidden * 2].view(torch.bfloat16).view(L, hidden)
    edges = []
    for e in (2 ** 31 // (2 * hidden), 2 ** 32 // (2 * hidden), 2 ** 31 // hidden):
        edges += [e - 1, e, e + 1]
    rows = np.unique(np.concatenate([np.arange(4), np.array(edges),
                                     random_rows(L, 40, seed=37).numpy(),
                                     np.arange(L - 8, L)])).astype(np.int64)
    ridx = torch.from_numpy(rows).to(DEV)
    r = orc.mlp_block(to64(x[ridx]), mod[rows], to64(sh), to64(sc), to64(gt), to64(w1), to64(w2))
    assert_parity(to64(h[ridx]), r["h"], f"mlp, L = {L}: h of the sampled rows")
    assert_parity(to64(out[ridx]), r["out"], f"mlp, L = {L}: out of the sampled rows",
                  bf16_storage=False)
    del ws, out, x, w1, w2, h
    torch.cuda.empty_cache()
