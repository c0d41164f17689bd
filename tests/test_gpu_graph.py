"""The fused block inside a CUDA graph.

Every entry point enqueues its kernels on the caller's stream and does no
host synchronisation (unless H3_DEBUG_SYNC is set), so a denoising loop can
capture one step into a CUDA graph and replay it ("Joint Audio-Video
Generation in Production", §4 Denoising Execution Flow: the same forward at
every step).  Captured after one plain call (which looks up the library's
per-device state), a step replays with the same bits as the direct call, and
a step captured in place (out aliasing x) replays as the sweep."""
import pytest
import torch

from h3inputs import CONFIGS, block_inputs
from tests.test_gpu_block import _layouts

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _setup(h3, name):
    c = CONFIGS[name]
    inp = block_inputs(c)
    mod, pos, _, _ = _layouts(h3, c)
    desc = h3.BlockDesc.make(L=c.L, d=c.d, n_heads=c.n_heads)
    nbytes = h3.h3_workspace_size(desc)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    dv = {k: v.to(DEV) for k, v in inp.items() if k != "x_raw"}
    dv["mod"] = torch.from_numpy(mod).to(DEV)
    dv["pos"] = torch.from_numpy(pos).to(DEV)
    return c, desc, nbytes, ws, dv


def _step(h3, desc, nbytes, ws, dv, x, out):
    h3.h3_attn_block_fwd(desc, x, dv["mod"], dv["pos"], dv["shift"], dv["scale"], dv["gate"],
                         dv["Wqkv"], dv["Wo"], ws, nbytes, out)


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_graph_replay_equals_direct_call(h3, name):
    c, desc, nbytes, ws, dv = _setup(h3, name)
    ref = torch.empty(c.L, c.d, dtype=torch.bfloat16, device=DEV)
    _step(h3, desc, nbytes, ws, dv, dv["x"], ref)          # plain call first
    assert h3.h3_sync_status() == 0
    out = torch.full_like(ref, float("nan"))
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            _step(h3, desc, nbytes, ws, dv, dv["x"], out)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert h3.h3_sync_status() == 0
        assert torch.equal(out.view(torch.uint8), ref.view(torch.uint8))


def test_graph_in_place_sweep_equals_direct_steps(h3):
    c, desc, nbytes, ws, dv = _setup(h3, "small")
    steps = 4
    x_direct = dv["x"].clone()
    for _ in range(steps):
        _step(h3, desc, nbytes, ws, dv, x_direct, x_direct)   # out aliases x: the sweep
    assert h3.h3_sync_status() == 0
    x_graph = dv["x"].clone()
    warm = dv["x"].clone()
    _step(h3, desc, nbytes, ws, dv, warm, warm)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            _step(h3, desc, nbytes, ws, dv, x_graph, x_graph)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(steps):
        g.replay()
    torch.cuda.synchronize()
    assert h3.h3_sync_status() == 0
    assert torch.equal(x_graph.view(torch.uint8), x_direct.view(torch.uint8))
