"""GPU parity of the whole sub-block (fused call and the five separate calls)
against the CPU fp64 oracle, on the seeded block workloads.

The fused call leaves the rotated qkv and the attention output O in its
workspace, so those intermediates are compared on their own as well as the
final output.  Large workloads compare sampled rows (the oracle's row-slice
protocol: keys and values for all L tokens, queries for the sampled rows).
"""
import math

import pytest
import torch

import oracle as orc
from h3inputs import CONFIGS, block_inputs, random_rows
from tests._parity import CHAIN_MAX_REL_RMS, assert_parity, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _layouts(h3, c):
    args = (c.n_text, c.video_t, c.video_h, c.video_w, c.audio_channels, c.audio_steps)
    mod, pos = h3.h3_build_packed_layout(*args)
    omod, opos = orc.packed_layout(*args)
    return mod, pos, omod, opos


def _run_fused(h3, c, inp, mod, pos, causal=False):
    L, d = c.L, c.d
    desc = h3.BlockDesc.make(L=L, d=d, n_heads=c.n_heads, causal=causal)
    nbytes = h3.h3_workspace_size(desc)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=DEV)
    out = torch.full((L, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    dev = {k: v.to(DEV) for k, v in inp.items() if k != "x_raw"}
    h3.h3_attn_block_fwd(desc, dev["x"], torch.from_numpy(mod).to(DEV),
                         torch.from_numpy(pos).to(DEV), dev["shift"], dev["scale"], dev["gate"],
                         dev["Wqkv"], dev["Wo"], ws, nbytes, out)
    assert h3.h3_sync_status() == 0
    off = (L * d * 2 + 255) // 256 * 256
    O = ws[:L * d * 2].view(torch.bfloat16).view(L, d)
    qkv = ws[off:off + L * 3 * d * 2].view(torch.bfloat16).view(L, 3 * d)
    return out, qkv, O


def _oracle_inputs(inp):
    return {k: to64(v) for k, v in inp.items() if k != "x_raw"}


@pytest.mark.parametrize("name,causal", [("tiny", False), ("tiny", True), ("small", False)])
def test_block_parity_full_rows(h3, name, causal):
    c = CONFIGS[name]
    inp = block_inputs(c)
    mod, pos, omod, opos = _layouts(h3, c)
    out, qkv, O = _run_fused(h3, c, inp, mod, pos, causal)
    o = _oracle_inputs(inp)
    r = orc.block(o["x"], omod, opos, o["shift"], o["scale"], o["gate"], o["Wqkv"], o["Wo"],
                  c.n_heads, causal=causal)
    assert_parity(to64(qkv), r["qkv"], f"{name} qkv (rotated)")
    # O inside the chain also carries the bf16 storage of y and of the rotated
    # q, k (each logit moves by ~2^-8 against the fp64 chain): the chain bound
    assert_parity(to64(O), r["O"], f"{name} O", max_rel_rms=CHAIN_MAX_REL_RMS)
    assert_parity(to64(out), r["out"], f"{name} out", bf16_storage=False)
    # the branch O Wo^T on its own (the residual dilutes its errors in out):
    # the output projection with a zero residual and a unit gate
    L, d = c.L, c.d
    br = torch.empty(L, d, dtype=torch.bfloat16, device=DEV)
    h3.h3_out_proj_gated_residual(O, inp["Wo"].to(DEV), torch.zeros_like(br),
                                  torch.zeros(L, dtype=torch.uint8, device=DEV),
                                  torch.ones(1, d, device=DEV), L, d, 1, br)
    assert h3.h3_sync_status() == 0
    assert_parity(to64(br), r["branch"], f"{name} branch O Wo^T",
                  max_rel_rms=CHAIN_MAX_REL_RMS)


def test_block_separate_calls_match_oracle(h3):
    """Route 2: modulate -> qkv_proj -> mrope -> attention -> out_proj."""
    c = CONFIGS["small"]
    inp = block_inputs(c)
    mod, pos, omod, opos = _layouts(h3, c)
    L, d, H = c.L, c.d, c.n_heads
    dev = {k: v.to(DEV) for k, v in inp.items() if k != "x_raw"}
    md, pd = torch.from_numpy(mod).to(DEV), torch.from_numpy(pos).to(DEV)
    y = torch.empty(L, d, dtype=torch.bfloat16, device=DEV)
    qkv = torch.empty(L, 3 * d, dtype=torch.bfloat16, device=DEV)
    O = torch.empty(L, d, dtype=torch.bfloat16, device=DEV)
    out = torch.empty(L, d, dtype=torch.bfloat16, device=DEV)
    h3.h3_adaln_modulate(dev["x"], md, dev["shift"], dev["scale"], L, d, 3, 1e-6, y)
    h3.h3_qkv_proj(y, dev["Wqkv"], L, d, qkv)
    h3.h3_mrope_apply(qkv, pd, L, H)
    h3.h3_joint_attn_fwd(qkv, L, H, 128, 0, 1 / math.sqrt(128), O)
    h3.h3_out_proj_gated_residual(O, dev["Wo"], dev["x"], md, dev["gate"], L, d, 3, out)
    assert h3.h3_sync_status() == 0
    o = _oracle_inputs(inp)
    r = orc.block(o["x"], omod, opos, o["shift"], o["scale"], o["gate"], o["Wqkv"], o["Wo"], H)
    assert_parity(to64(y), r["y"], "y")
    assert_parity(to64(qkv), r["qkv"], "qkv")
    assert_parity(to64(O), r["O"], "O", max_rel_rms=CHAIN_MAX_REL_RMS)
    assert_parity(to64(out), r["out"], "out", bf16_storage=False)


@pytest.mark.parametrize("causal", [False, True])
def test_block_parity_medium_sampled_rows(h3, causal):
    c = CONFIGS["medium"]
    inp = block_inputs(c)
    mod, pos, omod, opos = _layouts(h3, c)
    out, qkv, O = _run_fused(h3, c, inp, mod, pos, causal)
    rows = random_rows(c.L, 96, seed=7).numpy()
    o = _oracle_inputs(inp)
    r = orc.block_rows(o["x"], omod, opos, o["shift"], o["scale"], o["gate"], o["Wqkv"], o["Wo"],
                       rows, c.n_heads, causal=causal)
    d = c.d
    q = to64(qkv[torch.from_numpy(rows).to(DEV)])
    assert_parity(q[:, :d], r["q"], "medium q rows")
    assert_parity(to64(qkv[:, d:2 * d]), r["k"], "medium k (all rows)")
    assert_parity(to64(qkv[:, 2 * d:]), r["v"], "medium v (all rows)")
    assert_parity(to64(O[torch.from_numpy(rows).to(DEV)]), r["O"], "medium O rows",
                  max_rel_rms=CHAIN_MAX_REL_RMS)
    assert_parity(to64(out[torch.from_numpy(rows).to(DEV)]), r["out"], "medium out rows",
                  bf16_storage=False)


def test_block_deterministic(h3):
    c = CONFIGS["small"]
    inp = block_inputs(c)
    mod, pos, _, _ = _layouts(h3, c)
    a, _, _ = _run_fused(h3, c, inp, mod, pos)
    b, _, _ = _run_fused(h3, c, inp, mod, pos)
    assert torch.equal(a, b)


def test_block_gate_zero_returns_input(h3):
    c = CONFIGS["tiny"]
    inp = block_inputs(c)
    inp["gate"] = torch.zeros_like(inp["gate"])
    mod, pos, _, _ = _layouts(h3, c)
    out, _, _ = _run_fused(h3, c, inp, mod, pos)
    assert torch.equal(out.cpu(), inp["x"])


def test_block_widest_model_all_rows(h3):
    """The widest hidden size the library takes (d = 16,384: 128 heads; 3d =
    49,152 columns of Wqkv and of qkv) on a short ragged sequence, all rows
    against the oracle: row strides, the CTA-pair GEMM's 256-row tiles past a
    ragged M, and 128 attention heads."""
    from h3inputs import BlockConfig
    c = BlockConfig("widest", 21, 2, 5, 6, 2, 70, d=16384, n_heads=128, seed=17)
    assert c.L == 221
    inp = block_inputs(c)
    mod, pos, omod, opos = _layouts(h3, c)
    out, qkv, O = _run_fused(h3, c, inp, mod, pos)
    o = _oracle_inputs(inp)
    r = orc.block(o["x"], omod, opos, o["shift"], o["scale"], o["gate"], o["Wqkv"], o["Wo"],
                  c.n_heads)
    assert_parity(to64(qkv), r["qkv"], "widest qkv (rotated)")
    assert_parity(to64(O), r["O"], "widest O", max_rel_rms=CHAIN_MAX_REL_RMS)
    assert_parity(to64(out), r["out"], "widest out", bf16_storage=False)
