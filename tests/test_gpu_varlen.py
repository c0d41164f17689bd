"""GPU parity of block-diagonal (cu_seqlens) attention against the oracle
("Joint Audio-Video Generation in Production", §3 Packed Sequences and
Modality Identity Preservation: each token attends only within its own
sub-sequence; worked example cu_seqlens [0, 10, 30] and [0, 10, 30, 45])."""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from h3inputs import CONFIGS, attention_qkv, block_inputs, random_rows
from tests._parity import CHAIN_MAX_REL_RMS, assert_parity, assert_parity_rows, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCALE = 1 / math.sqrt(128)


def _run(h3, qkv, cu, H, causal):
    L = qkv.shape[0]
    O = torch.full((L, H * 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(H, L, dtype=torch.float32, device=DEV)
    h3.h3_joint_attn_varlen_fwd(qkv.to(DEV), cu, L, H, 128, causal, SCALE, O, lse)
    assert h3.h3_sync_status() == 0
    return O, lse


@pytest.mark.parametrize("cu,H,causal", [
    ([0, 10, 30], 1, 0), ([0, 10, 30, 45], 2, 0), ([0, 10, 30, 45], 1, 1),
    ([0, 7, 7, 130, 300, 301, 700], 2, 0), ([0, 7, 7, 130, 300, 301, 700], 1, 1),
    ([0, 256, 512, 1000], 1, 0), ([0, 1], 1, 0),
    ([0, 511, 513, 1025, 1537], 2, 0), ([0, 511, 513, 1025, 1537], 1, 1),
])
def test_varlen_parity(h3, cu, H, causal):
    """Each row is held to its own RMS: a row of a one- or two-token segment
    is of the order of |v| and carries the rounding of its bf16 weights at
    that scale, while the rows of long segments set the slice RMS
    (test_varlen_bound_cpu.py builds the kernel's rounding and shows the
    slice-wide bound failing for it on the [0, 511, 513, ...] case)."""
    L = cu[-1]
    qkv = attention_qkv(L, H, seed=L + len(cu))
    O, lse = _run(h3, qkv, cu, H, causal)
    ro, rl = orc.attention_varlen(to64(qkv), cu, H, 128, causal=bool(causal))
    assert_parity_rows(to64(O), ro, f"varlen {cu} causal={causal}")
    np.testing.assert_allclose(to64(lse), rl, atol=2e-2, rtol=1e-3)


def test_varlen_many_segments(h3):
    g = np.random.default_rng(5)
    L = 3000
    cuts = np.sort(g.choice(np.arange(1, L), size=39, replace=False))
    cu = [0] + [int(c) for c in cuts] + [L]
    qkv = attention_qkv(L, 1, seed=77)
    O, _ = _run(h3, qkv, cu, 1, 0)
    ro, _ = orc.attention_varlen(to64(qkv), cu, 1, 128)
    assert_parity(to64(O), ro, "varlen 40 segments")


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_varlen_modality_segments(h3, name):
    c = CONFIGS[name]
    cu = [0, c.n_text, c.n_text + c.n_video, c.L]
    qkv = attention_qkv(c.L, 2, seed=9)
    for causal in (0, 1):
        O, _ = _run(h3, qkv, cu, 2, causal)
        ro, _ = orc.attention_varlen(to64(qkv), cu, 2, 128, causal=bool(causal))
        assert_parity(to64(O), ro, f"{name} modality segments causal={causal}")


def test_one_segment_equals_full_attention_bitwise(h3):
    L, H = 777, 2
    qkv = attention_qkv(L, H, seed=3).to(DEV)
    a = torch.empty(L, H * 128, dtype=torch.bfloat16, device=DEV)
    b = torch.empty_like(a)
    h3.h3_joint_attn_fwd(qkv, L, H, 128, 0, SCALE, a)
    h3.h3_joint_attn_varlen_fwd(qkv, [0, L], L, H, 128, 0, SCALE, b)
    assert h3.h3_sync_status() == 0
    assert torch.equal(a, b)


@pytest.mark.parametrize("causal", [0, 1])
def test_varlen_full_size_modality_segments(h3, causal):
    c = CONFIGS["full"]
    cu = [0, c.n_text, c.n_text + c.n_video, c.L]
    qkv = attention_qkv(c.L, c.n_heads, seed=61)
    O, _ = _run(h3, qkv, cu, c.n_heads, causal)
    rows = np.unique(np.concatenate([random_rows(c.L, 40, seed=8).numpy(),
                                     np.array([0, 357, 358, 359, 57957, 57958, c.L - 1])]))
    ro, _ = orc.attention_varlen(to64(qkv), cu, c.n_heads, 128, causal=bool(causal), rows=rows)
    got = to64(O[torch.from_numpy(rows).to(DEV)])
    if causal:
        # a causal row of a segment sees the keys from the segment start to
        # itself (1 to 57,600): each row against its own RMS, as for causal rows
        assert_parity_rows(got, ro, "full-size modality segments, causal")
        return
    # segments are independent attention problems with very different output
    # scales (358 text keys vs 57,600 video keys): each is held to its own RMS
    seg = np.searchsorted(np.array(cu), rows, side="right") - 1
    for s in range(3):
        pick = seg == s
        assert pick.sum() >= 2
        assert_parity(got[pick], ro[pick], f"full-size modality segment {s}")


def test_block_with_segments(h3):
    c = CONFIGS["small"]
    cu = [0, c.n_text, c.n_text + c.n_video, c.L]
    inp = block_inputs(c)
    args = (c.n_text, c.video_t, c.video_h, c.video_w, c.audio_channels, c.audio_steps)
    mod, pos = h3.h3_build_packed_layout(*args)
    omod, opos = orc.packed_layout(*args)
    desc = h3.BlockDesc.make(L=c.L, d=c.d, n_heads=c.n_heads, cu_seqlens=cu)
    nbytes = h3.h3_workspace_size(desc)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    out = torch.empty(c.L, c.d, dtype=torch.bfloat16, device=DEV)
    dv = {k: v.to(DEV) for k, v in inp.items() if k != "x_raw"}
    h3.h3_attn_block_fwd(desc, dv["x"], torch.from_numpy(mod).to(DEV),
                         torch.from_numpy(pos).to(DEV), dv["shift"], dv["scale"], dv["gate"],
                         dv["Wqkv"], dv["Wo"], ws, nbytes, out)
    assert h3.h3_sync_status() == 0
    f = lambda k: to64(inp[k])
    r = orc.block(f("x"), omod, opos, f("shift"), f("scale"), f("gate"), f("Wqkv"), f("Wo"),
                  c.n_heads, cu_seqlens=cu)
    assert_parity(to64(out), r["out"], "block with modality segments", bf16_storage=False)
    O = ws[:c.L * c.d * 2].view(torch.bfloat16).view(c.L, c.d)
    assert_parity(to64(O), r["O"], "block O with modality segments", max_rel_rms=CHAIN_MAX_REL_RMS)
