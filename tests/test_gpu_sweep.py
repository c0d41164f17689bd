"""The denoising sweep: the sub-block run 50 times back to back on one stream,
each step with its own seeded per-modality shift/scale/gate (standing in for
the timestep) and the previous step's output as its input ("Joint Audio-Video
Generation in Production", §1: the attention over the packed sequence runs at
each of the 50 denoising steps; §4 Denoising Execution Flow).

The oracle runs its own 50-step chain (float64 inside a step, the step's
output stored as bf16 - the block's input/output type - before it becomes the
next input) at the tiny size and is compared at steps 1, 25 and 50.  At full
size the oracle takes the input of steps 1, 25 and 50 exactly as the GPU
consumed it (a bf16 state, like a seeded draw), computes that step itself on
the 1,024-row slice (keys and values of every token), and the step's output,
rotated qkv and O are compared with it; errors therefore do not compound
across steps, and every expected value is the oracle's own.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from h3inputs import CONFIGS, block_inputs, sweep_modulation
from tests._parity import assert_parity, to64
from tests.test_gpu_fullsize import check_full_block_slice

pytestmark = pytest.mark.gpu
DEV = "cuda"
STEPS = 50
CHECK = (1, 25, 50)


def _setup(h3, c):
    inp = block_inputs(c)
    args = (c.n_text, c.video_t, c.video_h, c.video_w, c.audio_channels, c.audio_steps)
    mod, pos = h3.h3_build_packed_layout(*args)
    desc = h3.BlockDesc.make(L=c.L, d=c.d, n_heads=c.n_heads)
    nbytes = h3.h3_workspace_size(desc)
    dev = {
        "x": inp["x"].to(DEV).clone(),
        "Wqkv": inp["Wqkv"].to(DEV), "Wo": inp["Wo"].to(DEV),
        "mod": torch.from_numpy(mod).to(DEV), "pos": torch.from_numpy(pos).to(DEV),
        "ws": torch.empty(nbytes, dtype=torch.uint8, device=DEV),
        "mods": [{k: v.to(DEV) for k, v in sweep_modulation(c, k).items()}
                 for k in range(1, STEPS + 1)],
    }
    return inp, desc, nbytes, dev


def _step(h3, desc, nbytes, dev, k, x, out):
    m = dev["mods"][k - 1]
    h3.h3_attn_block_fwd(desc, x, dev["mod"], dev["pos"], m["shift"], m["scale"], m["gate"],
                         dev["Wqkv"], dev["Wo"], dev["ws"], nbytes, out)


def _sweep(h3, desc, nbytes, dev, keep=CHECK, inner=False):
    """Run the sweep in place on a copy of dev['x']; return copies of the
    states at `keep` (and, with `inner`, of the rotated qkv and O those steps
    left in the workspace)."""
    x = dev["x"].clone()
    L, d = desc.L, desc.d
    off = (L * d * 2 + 255) // 256 * 256
    saved = {}
    for k in range(1, STEPS + 1):
        if k in keep:
            saved[f"in{k}"] = x.clone()
        _step(h3, desc, nbytes, dev, k, x, x)          # out aliases x
        if k in keep:
            saved[k] = x.clone()
            if inner:
                saved[f"O{k}"] = dev["ws"][:L * d * 2].view(torch.bfloat16).view(L, d).clone()
                saved[f"qkv{k}"] = dev["ws"][off:off + L * 3 * d * 2].view(
                    torch.bfloat16).view(L, 3 * d).clone()
    assert h3.h3_sync_status() == 0
    return saved


def test_sweep_tiny_against_oracle_chain(h3):
    c = CONFIGS["tiny"]
    inp, desc, nbytes, dev = _setup(h3, c)
    got = _sweep(h3, desc, nbytes, dev)
    omod, opos = orc.packed_layout(c.n_text, c.video_t, c.video_h, c.video_w,
                                   c.audio_channels, c.audio_steps)
    x = to64(inp["x"])
    wqkv, wo = to64(inp["Wqkv"]), to64(inp["Wo"])
    for k in range(1, STEPS + 1):
        m = {n: v.double().numpy() for n, v in sweep_modulation(c, k).items()}
        out = orc.block(x, omod, opos, m["shift"], m["scale"], m["gate"], wqkv, wo,
                        c.n_heads)["out"]
        # the step's output becomes the next input in the block's bf16 type
        x = torch.from_numpy(out).to(torch.bfloat16).double().numpy()
        if k in CHECK:
            # step 1 is one block: the plain bound.  Later steps compare two chains
            # whose bf16 states were rounded independently at every step before.
            if k == 1:
                assert_parity(to64(got[k]), out, f"sweep step {k}", bf16_storage=False)
            else:
                assert_parity(to64(got[k]), out, f"sweep step {k}",
                              roundings=3.0 * np.sqrt(k - 1))


def test_sweep_full_size_against_oracle_slice(h3):
    c = CONFIGS["full"]
    inp, desc, nbytes, dev = _setup(h3, c)
    a = _sweep(h3, desc, nbytes, dev, inner=True)
    omod, opos = orc.packed_layout(c.n_text, c.video_t, c.video_h, c.video_w,
                                   c.audio_channels, c.audio_steps)
    wqkv, wo = to64(inp["Wqkv"]), to64(inp["Wo"])
    for k in CHECK:
        # the state moves: each checked step differs from its input
        assert not torch.equal(a[k], a[f"in{k}"])
        m64 = {n: v.double().numpy() for n, v in sweep_modulation(c, k).items()}
        check_full_block_slice(c, to64(a[f"in{k}"]), omod, opos, m64, wqkv, wo, a[k],
                               a[f"qkv{k}"], a[f"O{k}"], f"sweep step {k}")
        for n in (f"O{k}", f"qkv{k}"):
            del a[n]
    # bitwise deterministic
    b = _sweep(h3, desc, nbytes, dev, keep=(50,))
    assert torch.equal(a[50], b[50])
