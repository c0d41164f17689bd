"""The checked build (libh3attn_checked.so, compiled with H3_CHECKED): every
global-memory load and store that a kernel addresses itself first tests its
row and column against its buffer's extents, and a failed test is reported
as H3_ERR_OUT_OF_BOUNDS instead of touching memory.  These tests run the same
calls through both libraries and require the checked one to report nothing
and to give bit-identical results (the checks change no arithmetic), and the
bounds self-test to be reported (its one access lies past a one-element
buffer and is skipped; nothing invalid reaches memory)."""
import contextlib
import math

import pytest
import torch

import joint_audio_video_gb300 as h3lib
from h3inputs import CONFIGS, attention_qkv, block_inputs
from tests.test_gpu_block import _layouts, _run_fused
from tests.test_gpu_fp8 import _run_fp8_block
from tests.test_gpu_mlp import _inputs as _mlp_inputs
from tests.test_gpu_mlp import _run as _run_mlp

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def checked(h3):
    from joint_audio_video_gb300 import build as b
    b.build(checked=True)
    lib = h3lib.load_checked()
    assert lib.h3_checked_build() == 1
    assert h3lib.h3_checked_build() is False
    return lib


@contextlib.contextmanager
def _through(lib):
    """Route the binding's calls to `lib` for the duration of the block."""
    saved = h3lib._lib
    h3lib._lib = lib
    try:
        yield
    finally:
        h3lib._lib = saved


def _both(checked, fn):
    """fn() through the library and through the checked library; the checked
    run must report H3_OK and give the same bits."""
    ref = fn()
    assert h3lib.h3_sync_status() == 0
    with _through(checked):
        got = fn()
        assert h3lib.h3_sync_status() == 0
    for a, b in zip(ref, got):
        assert torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.uint8) if b.dtype == torch.bfloat16 else b)


def test_bounds_selftest_is_reported_and_the_context_survives(checked):
    st = torch.cuda.current_stream().cuda_stream
    assert h3lib.h3_selftest_bounds_check() == 2          # normal build: launches nothing
    assert checked.h3_selftest_bounds_check(st) == 0
    assert checked.h3_sync_status(st) == 7                 # H3_ERR_OUT_OF_BOUNDS
    assert checked.h3_sync_status(st) == 0                 # read and cleared
    x = torch.ones(4, device=DEV)
    assert float((x * 2).sum()) == 8.0


@pytest.mark.parametrize("name,causal", [("tiny", True), ("small", False)])
def test_checked_block_matches(h3, checked, name, causal):
    c = CONFIGS[name]
    inp = block_inputs(c)
    mod, pos, _, _ = _layouts(h3, c)
    _both(checked, lambda: _run_fused(h3, c, inp, mod, pos, causal))


def test_checked_varlen_and_projections_match(h3, checked):
    L, H = 1000, 3          # d = 384: 3d is not a multiple of 256 (single-CTA GEMM form)
    d = H * 128
    qkv = attention_qkv(L, H, seed=31).to(DEV)
    cu = [0, 10, 30, 45, 600, 1000]
    g = torch.Generator().manual_seed(32)
    y = torch.randn(L, d, generator=g).to(torch.bfloat16).to(DEV)
    w = (torch.randn(3 * d, d, generator=g) / math.sqrt(d)).to(torch.bfloat16).to(DEV)
    pos = torch.randint(0, 50, (L, 3), generator=g, dtype=torch.int32).to(DEV)

    def run():
        o = torch.full((L, d), float("nan"), dtype=torch.bfloat16, device=DEV)
        h3lib.h3_joint_attn_varlen_fwd(qkv, cu, L, H, 128, 1, None, o)
        p = torch.empty(L, 3 * d, dtype=torch.bfloat16, device=DEV)
        h3lib.h3_qkv_proj(y, w, L, d, p)
        h3lib.h3_mrope_apply(p, pos, L, H)
        return o, p

    _both(checked, run)


def test_checked_mlp_fp8_and_denoise_match(h3, checked):
    c = CONFIGS["tiny"]
    hidden = 4 * c.d
    x, w1, w2, sh, sc, gt = _mlp_inputs(c, hidden, seed=33)
    mod, pos, _, _ = _layouts(h3, c)
    inp = block_inputs(c)
    L, C = c.L, 96
    g = torch.Generator().manual_seed(34)
    z0 = torch.randn(L, C, generator=g)
    v = torch.randn(L, C, generator=g).to(torch.bfloat16).to(DEV)
    md = torch.from_numpy(mod).to(DEV)

    def run():
        out, hmid = _run_mlp(h3lib, c, hidden, x, w1, w2, sh, sc, gt, mod)
        out8, qkv8, O8 = _run_fp8_block(h3lib, c, inp, mod, pos)
        z = z0.to(DEV)
        x0 = torch.empty_like(z)
        h3lib.h3_denoise_step(z, x0, v, md, None, None, L, C, [0.0, 0.5, 0.25],
                              [0.0, 0.25, 0.125], [0, 1, 1])
        return out, hmid, out8, qkv8, O8, z, x0

    _both(checked, run)
