"""Full-size parity: the packed sequence of 58,758 tokens (358 text + 57,600
video + 800 audio), d = 5120, 40 heads, in the launch configuration the
benchmark times.  The oracle computes sampled output rows one by one (keys and
values for all tokens, queries only for the sampled rows), including the
ragged 6-row tail that a 128-row tiling leaves at this length ("Joint
Audio-Video Generation in Production", §6 Boundary Trimming: exactly the
effective tokens, no padding)."""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from h3inputs import CONFIGS, attention_qkv, block_inputs, random_rows
from tests._parity import assert_parity, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"
CHAIN_MAX_REL_RMS = 4e-2


def _sample_rows(L, n, seed):
    rows = random_rows(L, n, seed).numpy()
    tail = np.arange(L - 8, L)                      # the ragged last tile
    text = np.arange(0, 4)
    return np.unique(np.concatenate([rows, tail, text]))


def test_full_attention_sampled_rows(h3):
    c = CONFIGS["full"]
    L, H = c.L, c.n_heads
    assert L % 128 == 6
    qkv = attention_qkv(L, H, seed=58)
    dev = qkv.to(DEV)
    O = torch.full((L, H * 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(H, L, dtype=torch.float32, device=DEV)
    h3.h3_joint_attn_fwd(dev, L, H, 128, 0, 1 / math.sqrt(128), O, lse)
    assert h3.h3_sync_status() == 0
    assert torch.isfinite(O.float()).all()
    rows = _sample_rows(L, 48, seed=3)
    q64 = to64(qkv)
    ro, rl = orc.attention(q64, H, 128, rows=rows)
    ridx = torch.from_numpy(rows).to(DEV)
    assert_parity(to64(O[ridx]), ro, "full-size attention rows")
    np.testing.assert_allclose(to64(lse[:, ridx]), rl, atol=2e-2, rtol=1e-3)


def test_full_block_sampled_rows(h3):
    c = CONFIGS["full"]
    L, d, H = c.L, c.d, c.n_heads
    inp = block_inputs(c)
    args = (c.n_text, c.video_t, c.video_h, c.video_w, c.audio_channels, c.audio_steps)
    mod, pos = h3.h3_build_packed_layout(*args)
    omod, opos = orc.packed_layout(*args)
    desc = h3.BlockDesc.make(L=L, d=d, n_heads=H)
    nbytes = h3.h3_workspace_size(desc)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    out = torch.full((L, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    dv = {k: v.to(DEV) for k, v in inp.items() if k != "x_raw"}
    h3.h3_attn_block_fwd(desc, dv["x"], torch.from_numpy(mod).to(DEV),
                         torch.from_numpy(pos).to(DEV), dv["shift"], dv["scale"], dv["gate"],
                         dv["Wqkv"], dv["Wo"], ws, nbytes, out)
    assert h3.h3_sync_status() == 0
    assert torch.isfinite(out.float()).all()
    off = (L * d * 2 + 255) // 256 * 256
    O = ws[:L * d * 2].view(torch.bfloat16).view(L, d)
    qkv = ws[off:off + L * 3 * d * 2].view(torch.bfloat16).view(L, 3 * d)
    rows = _sample_rows(L, 40, seed=4)
    f = lambda k: to64(inp[k])
    r = orc.block_rows(f("x"), omod, opos, f("shift"), f("scale"), f("gate"), f("Wqkv"),
                       f("Wo"), rows, H)
    ridx = torch.from_numpy(rows).to(DEV)
    assert_parity(to64(qkv[ridx, :d]), r["q"], "full q rows")
    krows = torch.from_numpy(np.arange(0, L, 97)).to(DEV)
    assert_parity(to64(qkv[krows, d:2 * d]), r["k"][np.arange(0, L, 97)], "full k rows")
    assert_parity(to64(qkv[krows, 2 * d:]), r["v"][np.arange(0, L, 97)], "full v rows")
    assert_parity(to64(O[ridx]), r["O"], "full O rows", max_rel_rms=CHAIN_MAX_REL_RMS)
    assert_parity(to64(out[ridx]), r["out"], "full out rows", bf16_storage=False)
