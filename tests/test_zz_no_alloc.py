"""The allocation-free fused entry point, h3_attn_block_fwd_noalloc.

It is for callers that cannot allocate device memory while they run (an
engine that fixes every device buffer before execution and passes its plugins
only their inputs and outputs, or a process whose caching allocator already
holds the GPU's memory): the library keeps a 64 MiB workspace per GPU for
them.  These checks call it through the C ABI twice in a row, on different
inputs, and compare each result with the allocating entry point's on the same
inputs, within the block-output tolerance the other tests use.  This file is
collected last so that a run stopping at its first failure has run every
other test.
"""
import pytest
import torch

from h3inputs import CONFIGS, block_inputs
from tests._parity import assert_parity, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _device_inputs(h3, c, seed):
    inp = block_inputs(c, seed=seed)
    mod, pos = h3.h3_build_packed_layout(c.n_text, c.video_t, c.video_h, c.video_w,
                                         c.audio_channels, c.audio_steps)
    d = {k: v.to(DEV) for k, v in inp.items() if k != "x_raw"}
    d["mod"] = torch.from_numpy(mod).to(DEV)
    d["pos"] = torch.from_numpy(pos).to(DEV)
    return d


def _args(d):
    return (d["x"], d["mod"], d["pos"], d["shift"], d["scale"], d["gate"], d["Wqkv"], d["Wo"])


def test_noalloc_matches_allocating_entry_point_twice(h3):
    c = CONFIGS["small"]                  # its workspace is exactly 64 MiB
    desc = h3.BlockDesc.make(L=c.L, d=c.d, n_heads=c.n_heads)
    need = h3.h3_workspace_size(desc)
    assert need <= h3.NOALLOC_SCRATCH_BYTES
    for seed in (101, 202):               # two calls in a row, different inputs
        d = _device_inputs(h3, c, seed)
        ws = torch.empty(need, dtype=torch.uint8, device=DEV)
        ref = torch.empty(c.L, c.d, dtype=torch.bfloat16, device=DEV)
        h3.h3_attn_block_fwd(desc, *_args(d), ws, need, ref)
        got = torch.full((c.L, c.d), float("nan"), dtype=torch.bfloat16, device=DEV)
        h3.h3_attn_block_fwd_noalloc(desc, *_args(d), got)
        assert h3.h3_sync_status() == 0
        assert_parity(to64(got), to64(ref), f"noalloc vs allocating (seed {seed})",
                      bf16_storage=False)


def test_noalloc_small_shape_after_large_one(h3):
    c = CONFIGS["tiny"]
    desc = h3.BlockDesc.make(L=c.L, d=c.d, n_heads=c.n_heads, causal=True)
    need = h3.h3_workspace_size(desc)
    d = _device_inputs(h3, c, 7)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    ref = torch.empty(c.L, c.d, dtype=torch.bfloat16, device=DEV)
    h3.h3_attn_block_fwd(desc, *_args(d), ws, need, ref)
    for _ in range(2):
        got = torch.full((c.L, c.d), float("nan"), dtype=torch.bfloat16, device=DEV)
        h3.h3_attn_block_fwd_noalloc(desc, *_args(d), got)
        assert h3.h3_sync_status() == 0
        assert_parity(to64(got), to64(ref), "noalloc tiny causal", bf16_storage=False)


def test_noalloc_rejects_shapes_beyond_its_workspace(h3):
    c = CONFIGS["full"]
    desc = h3.BlockDesc.make(L=c.L, d=c.d, n_heads=c.n_heads)
    assert h3.h3_workspace_size(desc) > h3.NOALLOC_SCRATCH_BYTES
    p = 1 << 20
    with pytest.raises(h3.H3Error) as e:
        h3.h3_attn_block_fwd_noalloc(desc, p, p, p, p, p, p, p, p, p + (1 << 30))
    assert e.value.status == 6            # H3_ERR_WORKSPACE, nothing launched
    assert h3.h3_sync_status() == 0
