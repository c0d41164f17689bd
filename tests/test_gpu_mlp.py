"""GPU parity of the MLP sub-block (second modality-modulated LayerNorm, the
feed-forward up projection with GELU, the down projection with the gated
residual) against the oracle ("DiffusionNFT on MiniMax H3": feed-forward
projections ff.net.0.proj and ff.net.2 beside the attention's; width 4d and
the tanh form of GELU are readings)."""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from h3inputs import CONFIGS, random_rows
from tests._parity import assert_parity, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(c, hidden, seed):
    g = torch.Generator().manual_seed(seed)
    L, d = c.L, c.d
    x = torch.randn(L, d, generator=g).to(torch.bfloat16)
    w1 = (torch.randn(hidden, d, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    w2 = (torch.randn(d, hidden, generator=g) / math.sqrt(hidden)).to(torch.bfloat16)
    sh, sc, gt = (torch.randn(3, d, generator=g) * 0.1 for _ in range(3))
    return x, w1, w2, sh, sc, gt


def _run(h3, c, hidden, x, w1, w2, sh, sc, gt, mod):
    desc = h3.MlpDesc.make(L=c.L, d=c.d, hidden=hidden)
    nbytes = h3.h3_mlp_workspace_size(desc)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    out = torch.full((c.L, c.d), float("nan"), dtype=torch.bfloat16, device=DEV)
    h3.h3_mlp_block_fwd(desc, x.to(DEV), torch.from_numpy(mod).to(DEV), sh.to(DEV), sc.to(DEV),
                        gt.to(DEV), w1.to(DEV), w2.to(DEV), ws, nbytes, out)
    assert h3.h3_sync_status() == 0
    off = (c.L * c.d * 2 + 255) // 256 * 256
    h = ws[off:off + c.L * hidden * 2].view(torch.bfloat16).view(c.L, hidden)
    return out, h


def _mod(h3, c):
    mod, _ = h3.h3_build_packed_layout(c.n_text, c.video_t, c.video_h, c.video_w,
                                       c.audio_channels, c.audio_steps)
    return mod


@pytest.mark.parametrize("name,hidden", [("tiny", 1024), ("tiny", 384), ("small", 8192)])
def test_mlp_block_parity(h3, name, hidden):
    c = CONFIGS[name]
    mod = _mod(h3, c)
    x, w1, w2, sh, sc, gt = _inputs(c, hidden, seed=hidden + c.L)
    out, h = _run(h3, c, hidden, x, w1, w2, sh, sc, gt, mod)
    r = orc.mlp_block(to64(x), mod, to64(sh), to64(sc), to64(gt), to64(w1), to64(w2))
    assert_parity(to64(h), r["h"], f"{name} mlp h")
    assert_parity(to64(out), r["out"], f"{name} mlp out", bf16_storage=False)


@pytest.mark.parametrize("name", ["medium", "full"])
def test_mlp_block_sampled_rows(h3, name):
    c = CONFIGS[name]
    hidden = 4 * c.d
    mod = _mod(h3, c)
    x, w1, w2, sh, sc, gt = _inputs(c, hidden, seed=7)
    out, h = _run(h3, c, hidden, x, w1, w2, sh, sc, gt, mod)
    rows = np.unique(np.concatenate([random_rows(c.L, 48, seed=2).numpy(),
                                     np.arange(c.L - 6, c.L)]))
    r = orc.mlp_block(to64(x[rows]), mod[rows], to64(sh), to64(sc), to64(gt), to64(w1),
                      to64(w2))
    ridx = torch.from_numpy(rows).to(DEV)
    assert_parity(to64(h[ridx]), r["h"], f"{name} mlp h rows")
    assert_parity(to64(out[ridx]), r["out"], f"{name} mlp out rows", bf16_storage=False)


def test_mlp_gate_zero_returns_input(h3):
    c = CONFIGS["tiny"]
    mod = _mod(h3, c)
    x, w1, w2, sh, sc, gt = _inputs(c, 1024, seed=1)
    out, _ = _run(h3, c, 1024, x, w1, w2, sh, sc, torch.zeros_like(gt), mod)
    assert torch.equal(out.cpu(), x)
