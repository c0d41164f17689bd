"""Full-size parity: the packed sequence of 58,758 tokens (358 text + 57,600
video + 800 audio), d = 5120, 40 heads, in the launch configuration the
benchmark times.  The oracle computes a 1,024-row slice one row at a time:
keys and values for all tokens, queries for rows 0..127 (text), one video row
every 75 tokens (every latent frame) and the last 128 rows (audio, including
the ragged 6-row tail that a 128-row tiling leaves at this length; "Joint
Audio-Video Generation in Production", §6 Boundary Trimming: exactly the
effective tokens take part, nothing is padded)."""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from h3inputs import CONFIGS, attention_qkv, block_inputs, random_rows
from tests._parity import CHAIN_MAX_REL_RMS, assert_parity, assert_parity_rows, slice_rows, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_full_attention_slice_rows(h3):
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
    rows = slice_rows(L, c.n_text)
    ro, rl = orc.attention(to64(qkv), H, 128, rows=rows)
    ridx = torch.from_numpy(rows).to(DEV)
    assert_parity(to64(O[ridx]), ro, "full-size attention, slice rows")
    np.testing.assert_allclose(to64(lse[:, ridx]), rl, atol=2e-2, rtol=1e-3)


def test_full_causal_attention_slice_rows(h3):
    """The causal option at full length on the same slice: each row sees the
    keys up to itself in packed order ("多模态强化学习工程解析…", 三 目标模型),
    so the slice's rows see from one key (row 0) to all 58,758 (the last
    row), and every row's last key block is cut by the diagonal.  Each row is
    held to its own RMS (test_causal_bound_cpu.py shows why the slice-wide
    RMS cannot hold for the rows with a few keys)."""
    c = CONFIGS["full"]
    L, H = c.L, c.n_heads
    qkv = attention_qkv(L, H, seed=57)
    dev = qkv.to(DEV)
    O = torch.full((L, H * 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(H, L, dtype=torch.float32, device=DEV)
    h3.h3_joint_attn_fwd(dev, L, H, 128, 1, 1 / math.sqrt(128), O, lse)
    assert h3.h3_sync_status() == 0
    assert torch.isfinite(O.float()).all()
    rows = slice_rows(L, c.n_text)
    ro, rl = orc.attention(to64(qkv), H, 128, causal=True, rows=rows)
    ridx = torch.from_numpy(rows).to(DEV)
    assert_parity_rows(to64(O[ridx]), ro, "full-size causal attention, slice rows")
    np.testing.assert_allclose(to64(lse[:, ridx]), rl, atol=2e-2, rtol=1e-3)


def run_full_block(h3, c, x, shift, scale, gate, Wqkv, Wo, mod, pos):
    """One fused block at full size; returns out, the rotated qkv and O (both
    left in the block's workspace)."""
    L, d, H = c.L, c.d, c.n_heads
    desc = h3.BlockDesc.make(L=L, d=d, n_heads=H)
    nbytes = h3.h3_workspace_size(desc)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    out = torch.full((L, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    h3.h3_attn_block_fwd(desc, x, mod, pos, shift, scale, gate, Wqkv, Wo, ws, nbytes, out)
    assert h3.h3_sync_status() == 0
    off = (L * d * 2 + 255) // 256 * 256
    O = ws[:L * d * 2].view(torch.bfloat16).view(L, d)
    qkv = ws[off:off + L * 3 * d * 2].view(torch.bfloat16).view(L, 3 * d)
    return out, qkv, O


def check_full_block_slice(c, x64, mod, pos, m64, Wqkv64, Wo64, out, qkv, O, what):
    """The block's outputs on the 1,024-row slice against the oracle (K and V
    on every row, since the oracle forms them for all tokens anyway)."""
    L, d, H = c.L, c.d, c.n_heads
    rows = slice_rows(L, c.n_text)
    r = orc.block_rows(x64, mod, pos, m64["shift"], m64["scale"], m64["gate"], Wqkv64, Wo64,
                       rows, H)
    ridx = torch.from_numpy(rows).to(DEV)
    assert_parity(to64(qkv[ridx, :d]), r["q"], f"{what}: q, slice rows")
    assert_parity(to64(qkv[:, d:2 * d]), r["k"], f"{what}: k, all rows")
    assert_parity(to64(qkv[:, 2 * d:]), r["v"], f"{what}: v, all rows")
    assert_parity(to64(O[ridx]), r["O"], f"{what}: O, slice rows", max_rel_rms=CHAIN_MAX_REL_RMS)
    assert torch.isfinite(out.float()).all()
    assert_parity(to64(out[ridx]), r["out"], f"{what}: out, slice rows", bf16_storage=False)


def test_full_block_slice_rows(h3):
    c = CONFIGS["full"]
    inp = block_inputs(c)
    args = (c.n_text, c.video_t, c.video_h, c.video_w, c.audio_channels, c.audio_steps)
    mod, pos = h3.h3_build_packed_layout(*args)
    omod, opos = orc.packed_layout(*args)
    dv = {k: v.to(DEV) for k, v in inp.items() if k != "x_raw"}
    out, qkv, O = run_full_block(h3, c, dv["x"], dv["shift"], dv["scale"], dv["gate"],
                                 dv["Wqkv"], dv["Wo"], torch.from_numpy(mod).to(DEV),
                                 torch.from_numpy(pos).to(DEV))
    m64 = {k: to64(inp[k]) for k in ("shift", "scale", "gate")}
    check_full_block_slice(c, to64(inp["x"]), omod, opos, m64, to64(inp["Wqkv"]),
                           to64(inp["Wo"]), out, qkv, O, "full block")


# ---------------------------------------------------------------------------
# Moves of the running maximum at full length.  The kernel computes a block's
# exponentials against the row's running maximum and redoes the block when
# its maximum exceeds that by more than 8 (log2 units).  With unit-variance
# scores that never happens after the first blocks, so four heads are
# planted: in head 0 a group of query rows meets a ramp over the last 2,000
# keys (the maximum moves several times, late), in head 1 the same rows meet
# 6 large keys that sit in the masked tail block alone, and in heads 2 and 3
# they meet one key ~100 log2 units above everything before it, in the first
# and in the second half of a late block (the exponentials of the first pass
# over such a block reach 2^100).  Whether a row takes each path is worked
# out below from the inputs.
# ---------------------------------------------------------------------------
RESCALE_LOG2 = 8.0
BIG_LOG2 = 64.0


def _block_maxima(qkv64, H, rows, causal, sm_scale, h, width):
    """Per row: maxima (log2 units) of consecutive key groups of `width`."""
    L = qkv64.shape[0]
    d = H * 128
    q = qkv64[rows, h * 128:(h + 1) * 128]
    k = qkv64[:, d + h * 128:d + (h + 1) * 128]
    s = (q @ k.T) * (sm_scale / math.log(2.0))
    if causal:
        s = np.where(np.arange(L)[None, :] <= rows[:, None], s, -np.inf)
    n = (L + width - 1) // width
    pad = np.full((len(rows), n * width - L), -np.inf)
    return np.concatenate([s, pad], axis=1).reshape(len(rows), n, width).max(axis=2)


def _rescale_events(qkv64, H, rows, causal, sm_scale):
    """Per (head, row): how many key blocks move the running maximum by more
    than 8 (log2 units) over the maximum of everything before them."""
    ev = np.zeros((H, len(rows)), dtype=np.int64)
    for h in range(H):
        bm = _block_maxima(qkv64, H, rows, causal, sm_scale, h, 128)
        m = np.full(len(rows), -np.inf)
        for b in range(bm.shape[1]):
            fresh = np.isinf(m)
            move = ~fresh & (bm[:, b] > m + RESCALE_LOG2)
            ev[h] += move
            m = np.where(fresh | move, np.maximum(m, bm[:, b]), m)
    return ev


def _largest_jump(qkv64, H, rows, causal, sm_scale, h):
    """Per row: the largest amount (log2 units) by which a 64-key half block
    exceeds the maximum of all keys before it."""
    hm = _block_maxima(qkv64, H, rows, causal, sm_scale, h, 64)
    before = np.maximum.accumulate(np.concatenate(
        [np.full((len(rows), 1), -np.inf), hm[:, :-1]], axis=1), axis=1)
    with np.errstate(invalid="ignore"):
        jump = np.where(np.isinf(before), -np.inf, hm - before)
    return jump.max(axis=1)


@pytest.mark.parametrize("causal", [False, True])
def test_full_attention_running_maximum_moves(h3, causal):
    L, H = CONFIGS["full"].L, 4
    d = H * 128
    base = attention_qkv(L, H, seed=59).float()
    planted = random_rows(L, 160, seed=60).numpy()
    planted = np.unique(np.concatenate([planted, np.arange(L - 40, L)]))
    pin = torch.from_numpy(planted)
    # head 0: queries of the planted rows point along dims 0..7, keys ramp up along them
    ramp = torch.linspace(0.0, 7.0, 2000)
    base[L - 2000:, d + 0:d + 8] += ramp[:, None]
    base[pin, 0:8] += 4.0
    # head 1: only the 6 keys of the last (ragged) block carry the large component
    base[L - 6:, d + 128:d + 136] += 6.0
    base[pin, 128:136] += 4.0
    # heads 2 and 3: one key far above all others, in the first half (column 10)
    # and in the second half (column 100) of the fifth block from the end
    kb = ((L + 127) // 128 - 5) * 128
    base[kb + 10, d + 256:d + 264] += 10.0
    base[pin, 256:264] += 10.0
    base[kb + 100, d + 384:d + 392] += 10.0
    base[pin, 384:392] += 10.0
    qkv = base.to(torch.bfloat16)
    q64 = to64(qkv)
    sm = 1 / math.sqrt(128)
    ev = _rescale_events(q64, H, planted, causal, sm)
    late = planted >= L - 2000
    assert late.sum() >= 40
    # the inputs really drive the rows through each path: several moves in
    # head 0 for every planted row that sees the ramp, one in head 1 for every
    # row that sees the tail block, a jump above 64 in heads 2 and 3 for every
    # row that sees the planted key
    seen0 = planted >= L - 1000 if causal else np.ones_like(late)
    assert np.all(ev[0][seen0] >= 2), ev[0][seen0].min()
    seen1 = planted >= L - 6 if causal else np.ones_like(late)
    assert np.all(ev[1][seen1] >= 1)
    for h, col in ((2, kb + 10), (3, kb + 100)):
        seen = planted >= col if causal else np.ones_like(late)
        assert seen.sum() >= 40
        jump = _largest_jump(q64, H, planted[seen], causal, sm, h)
        assert np.all(jump > BIG_LOG2 + 8), jump.min()
    O = torch.full((L, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(H, L, dtype=torch.float32, device=DEV)
    h3.h3_joint_attn_fwd(qkv.to(DEV), L, H, 128, int(causal), sm, O, lse)
    assert h3.h3_sync_status() == 0
    rows = np.unique(np.concatenate([planted, random_rows(L, 64, seed=61).numpy()]))
    ro, rl = orc.attention(q64, H, 128, causal=causal, sm_scale=sm, rows=rows)
    ridx = torch.from_numpy(rows).to(DEV)
    assert_parity(to64(O[ridx]), ro, f"running-maximum rows (causal={causal})")
    np.testing.assert_allclose(to64(lse[:, ridx]), rl, atol=2e-2, rtol=1e-3)
