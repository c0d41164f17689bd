"""GPU parity of every C-ABI call against the CPU fp64 oracle.

Inputs are seeded (h3inputs); the oracle gets the same bf16 values widened to
float64.  Outputs are NaN-prefilled (an unwritten element fails the
finiteness check) and surrounded by guard bands (an out-of-range write fails
the canary check).  Shapes span several tiles and ragged tails.
"""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from h3inputs import CONFIGS, attention_qkv
from tests._parity import assert_parity, to64

pytestmark = pytest.mark.gpu

DEV = "cuda"
CANARY = 0x5A


class Guarded:
    """A device tensor with 4 KB canary bands on both sides."""

    def __init__(self, shape, dtype, fill=float("nan")):
        n = int(np.prod(shape))
        esz = torch.empty((), dtype=dtype).element_size()
        self.pad = 4096 // esz
        self.raw = torch.empty(n + 2 * self.pad, dtype=dtype, device=DEV)
        self.raw.view(torch.uint8).fill_(CANARY)
        self.t = self.raw[self.pad:self.pad + n].view(*shape)
        self.t.fill_(fill)

    def check(self):
        b = self.raw.view(torch.uint8)
        nb = self.pad * self.raw.element_size()
        assert int((b[:nb] != CANARY).sum()) == 0, "write before the buffer"
        assert int((b[-nb:] != CANARY).sum()) == 0, "write past the end of the buffer"


def _sync(h3):
    assert h3.h3_sync_status() == 0


# --------------------------------------------------------------------- modulate
@pytest.mark.parametrize("L,d", [(1, 128), (7, 384), (64, 256), (513, 2048), (97, 5120),
                                 (33, 16384)])
def test_adaln_modulate_parity(h3, L, d):
    g = torch.Generator().manual_seed(L * 7 + d)
    x = (torch.randn(L, d, generator=g) * 2 + 0.5).to(torch.bfloat16)
    mod = torch.randint(0, 3, (L,), generator=g, dtype=torch.uint8)
    shift = torch.randn(3, d, generator=g) * 0.1
    scale = torch.randn(3, d, generator=g) * 0.1
    y = Guarded((L, d), torch.bfloat16)
    xd, md, shd, scd = x.to(DEV), mod.to(DEV), shift.to(DEV), scale.to(DEV)
    h3.h3_adaln_modulate(xd, md, shd, scd, L, d, 3, 1e-6, y.t)
    _sync(h3)
    y.check()
    ref = orc.adaln_modulate(to64(x), mod.numpy(), to64(shift), to64(scale), 1e-6)
    assert_parity(to64(y.t), ref, f"adaln L={L} d={d}")


def test_adaln_modality_indexing_bit_exact(h3):
    """scale = -1 makes y = shift[mod[n]] exactly, whatever x is."""
    L, d = 300, 512
    g = torch.Generator().manual_seed(3)
    x = torch.randn(L, d, generator=g).to(torch.bfloat16).to(DEV)
    mod = torch.randint(0, 3, (L,), generator=g, dtype=torch.uint8)
    consts = torch.tensor([0.5, -1.25, 3.0])        # bf16-exact
    shift = consts[:, None].repeat(1, d).to(DEV)
    scale = torch.full((3, d), -1.0, device=DEV)
    y = torch.empty(L, d, dtype=torch.bfloat16, device=DEV)
    h3.h3_adaln_modulate(x, mod.to(DEV), shift, scale, L, d, 3, 1e-6, y)
    _sync(h3)
    want = consts[mod.long()][:, None].expand(L, d).to(torch.bfloat16)
    assert torch.equal(y.cpu(), want)


def test_adaln_bad_modality_flags_status(h3):
    L, d = 4, 256
    x = torch.randn(L, d, device=DEV).to(torch.bfloat16)
    mod = torch.tensor([0, 1, 7, 2], dtype=torch.uint8, device=DEV)
    z = torch.zeros(3, d, device=DEV)
    y = torch.zeros(L, d, dtype=torch.bfloat16, device=DEV)
    h3.h3_adaln_modulate(x, mod, z, z, L, d, 3, 1e-6, y)
    assert h3.h3_sync_status() == 5
    assert torch.isnan(y[2].float()).all() and torch.isfinite(y[[0, 1, 3]].float()).all()
    assert h3.h3_sync_status() == 0          # the status word was cleared


# --------------------------------------------------------------------- projection
@pytest.mark.parametrize("L,d", [(1, 128), (63, 256), (64, 256), (65, 256), (129, 384),
                                 (1000, 256), (300, 2048),
                                 # CTA-pair tiles (N % 256 == 0) with one row, and one
                                 # row past a 256-row pair tile
                                 (1, 256), (257, 512)])
def test_qkv_proj_parity(h3, L, d):
    g = torch.Generator().manual_seed(L + 11 * d)
    y = torch.randn(L, d, generator=g).to(torch.bfloat16)
    w = (torch.randn(3 * d, d, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    out = Guarded((L, 3 * d), torch.bfloat16)
    h3.h3_qkv_proj(y.to(DEV), w.to(DEV), L, d, out.t)
    _sync(h3)
    out.check()
    assert_parity(to64(out.t), orc.linear(to64(y), to64(w)), f"qkv_proj L={L} d={d}")


# --------------------------------------------------------------------- rope
@pytest.mark.parametrize("name,H", [("tiny", 2), ("small", 3)])
def test_mrope_parity(h3, name, H):
    c = CONFIGS[name]
    mod, pos = h3.h3_build_packed_layout(c.n_text, c.video_t, c.video_h, c.video_w,
                                         c.audio_channels, c.audio_steps)
    L = len(mod)
    qkv = attention_qkv(L, H, seed=5)
    dev = qkv.to(DEV)
    h3.h3_mrope_apply(dev, torch.from_numpy(pos).to(DEV), L, H)
    _sync(h3)
    _, opos = orc.packed_layout(c.n_text, c.video_t, c.video_h, c.video_w, c.audio_channels,
                                c.audio_steps)
    ref = orc.mrope(to64(qkv), opos, H)
    d = H * 128
    got = to64(dev)
    assert_parity(got[:, :2 * d], ref[:, :2 * d], f"mrope {name}")
    assert np.array_equal(got[:, 2 * d:], ref[:, 2 * d:])          # V untouched


def test_mrope_large_positions(h3):
    L, H = 257, 1
    g = torch.Generator().manual_seed(9)
    pos = torch.randint(0, 60000, (L, 3), generator=g, dtype=torch.int32)
    qkv = attention_qkv(L, H, seed=6)
    dev = qkv.to(DEV)
    h3.h3_mrope_apply(dev, pos.to(DEV), L, H)
    _sync(h3)
    ref = orc.mrope(to64(qkv), pos.numpy(), H)
    assert_parity(to64(dev)[:, :256], ref[:, :256], "mrope large positions")


# --------------------------------------------------------------------- attention
@pytest.mark.parametrize("L,H,causal", [(1, 1, 0), (5, 2, 0), (127, 1, 0), (128, 2, 0),
                                        (129, 1, 0), (255, 2, 0), (256, 1, 0), (257, 2, 0),
                                        (1000, 2, 0), (1, 1, 1), (129, 2, 1), (300, 1, 1),
                                        (600, 2, 1),
                                        # a CTA pair covers 512 query rows: one full
                                        # pair, one query row into the next pair (whose
                                        # second CTA has no rows), one into its second CTA
                                        (511, 1, 0), (512, 2, 0), (513, 1, 0), (769, 1, 0),
                                        (1025, 2, 0), (513, 2, 1), (769, 1, 1), (1025, 1, 1)])
def test_attention_parity(h3, L, H, causal):
    qkv = attention_qkv(L, H, seed=L + H)
    O = Guarded((L, H * 128), torch.bfloat16)
    lse = Guarded((H, L), torch.float32)
    h3.h3_joint_attn_fwd(qkv.to(DEV), L, H, 128, causal, 1 / math.sqrt(128), O.t, lse.t)
    _sync(h3)
    O.check()
    lse.check()
    ro, rl = orc.attention(to64(qkv), H, 128, causal=bool(causal))
    assert_parity(to64(O.t), ro, f"attention L={L} H={H} causal={causal}")
    np.testing.assert_allclose(to64(lse.t), rl, atol=2e-2, rtol=1e-3)


@pytest.mark.parametrize("qk_std", [0.3, 2.0, 4.0])
def test_attention_softmax_sharpness(h3, qk_std):
    """Flat to very peaked score rows (the lazy-rescale path moves the max)."""
    L, H = 700, 1
    qkv = attention_qkv(L, H, seed=21, qk_std=qk_std)
    O = torch.full((L, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    h3.h3_joint_attn_fwd(qkv.to(DEV), L, H, 128, 0, 1 / math.sqrt(128), O)
    _sync(h3)
    ro, _ = orc.attention(to64(qkv), H, 128)
    assert_parity(to64(O), ro, f"attention qk_std={qk_std}")


def test_attention_identical_keys_give_mean_of_values(h3):
    L, H = 333, 1
    qkv = attention_qkv(L, H, seed=4)
    qkv[:, 128:256] = qkv[0:1, 128:256]
    O = torch.empty(L, 128, dtype=torch.bfloat16, device=DEV)
    h3.h3_joint_attn_fwd(qkv.to(DEV), L, H, 128, 0, 1 / math.sqrt(128), O)
    _sync(h3)
    want = to64(qkv)[:, 256:].mean(axis=0)
    assert_parity(to64(O), np.tile(want, (L, 1)), "identical keys")


# --------------------------------------------------------------------- output projection
@pytest.mark.parametrize("L,d", [(1, 128), (65, 256), (129, 384), (700, 2048), (1, 256),
                                 (257, 512)])
def test_out_proj_gated_residual_parity(h3, L, d):
    g = torch.Generator().manual_seed(L * 3 + d)
    O = torch.randn(L, d, generator=g).to(torch.bfloat16)
    wo = (torch.randn(d, d, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    x = torch.randn(L, d, generator=g).to(torch.bfloat16)
    mod = torch.randint(0, 3, (L,), generator=g, dtype=torch.uint8)
    gate = torch.randn(3, d, generator=g) * 0.5
    out = Guarded((L, d), torch.bfloat16)
    h3.h3_out_proj_gated_residual(O.to(DEV), wo.to(DEV), x.to(DEV), mod.to(DEV), gate.to(DEV),
                                  L, d, 3, out.t)
    _sync(h3)
    out.check()
    ref = orc.gated_residual(to64(x), orc.linear(to64(O), to64(wo)), mod.numpy(), to64(gate))
    assert_parity(to64(out.t), ref, f"out_proj L={L} d={d}")


def test_out_proj_gate_zero_returns_residual_bit_exact(h3):
    L, d = 200, 256
    g = torch.Generator().manual_seed(1)
    O = torch.randn(L, d, generator=g).to(torch.bfloat16).to(DEV)
    wo = torch.randn(d, d, generator=g).to(torch.bfloat16).to(DEV)
    x = torch.randn(L, d, generator=g).to(torch.bfloat16).to(DEV)
    mod = torch.randint(0, 3, (L,), generator=g, dtype=torch.uint8).to(DEV)
    out = torch.empty_like(x)
    h3.h3_out_proj_gated_residual(O, wo, x, mod, torch.zeros(3, d, device=DEV), L, d, 3, out)
    _sync(h3)
    assert torch.equal(out, x)
    # in place on the residual
    x2 = x.clone()
    h3.h3_out_proj_gated_residual(O, wo, x2, mod, torch.zeros(3, d, device=DEV), L, d, 3, x2)
    _sync(h3)
    assert torch.equal(x2, x)


def test_out_proj_gate_indexing_bit_exact(h3):
    """Wo = I, O = 1, x = 0: out[n] = gate[mod[n]] exactly (bf16-exact gates)."""
    L, d = 130, 256
    g = torch.Generator().manual_seed(2)
    mod = torch.randint(0, 3, (L,), generator=g, dtype=torch.uint8)
    consts = torch.tensor([0.25, -2.0, 8.0])
    gate = consts[:, None].repeat(1, d)
    O = torch.ones(L, d, dtype=torch.bfloat16, device=DEV)
    wo = torch.eye(d, dtype=torch.bfloat16, device=DEV)
    x = torch.zeros(L, d, dtype=torch.bfloat16, device=DEV)
    out = torch.empty_like(x)
    h3.h3_out_proj_gated_residual(O, wo, x, mod.to(DEV), gate.to(DEV), L, d, 3, out)
    _sync(h3)
    assert torch.equal(out.cpu(), consts[mod.long()][:, None].expand(L, d).to(torch.bfloat16))


# --------------------------------------------------------------------- bounded waits
def test_bounded_wait_times_out_and_context_survives(h3):
    h3.h3_selftest_wait_timeout(2_000_000)      # 2 ms
    assert h3.h3_sync_status() == 4
    assert h3.h3_sync_status() == 0
    # the context is still usable
    L, d = 3, 128
    x = torch.randn(L, d, device=DEV).to(torch.bfloat16)
    z = torch.zeros(3, d, device=DEV)
    y = torch.empty_like(x)
    h3.h3_adaln_modulate(x, torch.zeros(L, dtype=torch.uint8, device=DEV), z, z, L, d, 3, 0.0, y)
    _sync(h3)
    assert torch.isfinite(y.float()).all()
