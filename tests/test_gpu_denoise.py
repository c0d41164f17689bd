"""GPU parity of the denoising-step update (RF v -> X0, eta = 0 Euler on
per-modality schedules, anchor re-pin) against the oracle ("Joint Audio-Video
Generation in Production", §4 Denoising Execution Flow; H3 time t = 1 - sigma
with the velocity sign reversed, "多模态强化学习工程解析…" 5.1)."""
import numpy as np
import pytest
import torch

import oracle as orc
from h3inputs import CONFIGS
from tests._parity import to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _layout(h3, c):
    mod, _ = h3.h3_build_packed_layout(c.n_text, c.video_t, c.video_h, c.video_w,
                                       c.audio_channels, c.audio_steps)
    return mod


def test_denoise_parity_full_size(h3):
    c = CONFIGS["full"]
    L, C = c.L, 96
    g = torch.Generator().manual_seed(31)
    mod = _layout(h3, c)
    z = torch.randn(L, C, generator=g)
    v = torch.randn(L, C, generator=g).to(torch.bfloat16)
    za = torch.randn(L, C, generator=g)
    anchor = (torch.rand(L, generator=g) < 0.05).to(torch.uint8)
    sigma, sigma_next, update = [0.0, 0.62, 0.41], [0.0, 0.5, 0.3], [0, 1, 1]
    zd, x0 = z.to(DEV), torch.full((L, C), float("nan"), device=DEV)
    h3.h3_denoise_step(zd, x0, v.to(DEV), torch.from_numpy(mod).to(DEV), anchor.to(DEV),
                       za.to(DEV), L, C, sigma, sigma_next, update)
    assert h3.h3_sync_status() == 0
    rz, rx = orc.denoise_step(to64(z), to64(v), mod, sigma, sigma_next, update,
                              anchor.numpy(), to64(za))
    gz, gx = to64(zd), to64(x0)
    # fp32 fused multiply-add of bf16/fp32 inputs: within a few fp32 ulps
    np.testing.assert_allclose(gz, rz, rtol=2e-7, atol=2e-7)
    np.testing.assert_allclose(gx, rx, rtol=2e-7, atol=2e-7)
    a = anchor.numpy().astype(bool)
    t = mod == 0
    assert np.array_equal(gz[a], to64(za)[a]) and np.array_equal(gx[a], to64(za)[a])
    assert np.array_equal(gz[t & ~a], to64(z)[t & ~a])


def test_denoise_three_step_trace_is_exact(h3):
    """bf16-exact x0 and noise, dyadic schedules: three steps land on x0 exactly."""
    c = CONFIGS["tiny"]
    L, C = c.L, 16
    mod = _layout(h3, c)
    g = torch.Generator().manual_seed(32)
    x0 = torch.randint(-32, 33, (L, C), generator=g).float() / 8
    eps = torch.randint(-32, 33, (L, C), generator=g).float() / 8
    anchor = torch.zeros(L, dtype=torch.uint8)
    anchor[[20, 40]] = 1
    za = torch.randint(-8, 9, (L, C), generator=g).float()
    sched = {1: [1.0, 0.75, 0.375, 0.0], 2: [1.0, 0.5, 0.25, 0.0]}
    z = eps.clone()
    z[anchor.bool()] = za[anchor.bool()]
    zd = z.to(DEV)
    v_h3 = (x0 - eps).to(torch.bfloat16).to(DEV)      # exact in bf16
    for k in range(3):
        s = [0.0, sched[1][k], sched[2][k]]
        sn = [0.0, sched[1][k + 1], sched[2][k + 1]]
        h3.h3_denoise_step(zd, None, v_h3, torch.from_numpy(mod).to(DEV), anchor.to(DEV),
                           za.to(DEV), L, C, s, sn, [0, 1, 1])
    assert h3.h3_sync_status() == 0
    got = zd.cpu()
    free = torch.from_numpy(mod > 0) & ~anchor.bool()
    assert torch.equal(got[free], x0[free])
    assert torch.equal(got[anchor.bool()], za[anchor.bool()])
    assert torch.equal(got[torch.from_numpy(mod == 0)], eps[torch.from_numpy(mod == 0)])


def test_denoise_bad_modality_is_reported(h3):
    L, C = 4, 8
    z = torch.ones(L, C, device=DEV)
    v = torch.ones(L, C, dtype=torch.bfloat16, device=DEV)
    mod = torch.tensor([1, 9, 1, 2], dtype=torch.uint8, device=DEV)
    h3.h3_denoise_step(z, None, v, mod, None, None, L, C, [0.0, 0.5, 0.5], [0.0, 0.25, 0.25],
                       [0, 1, 1])
    assert h3.h3_sync_status() == 5
    assert torch.equal(z[1].cpu(), torch.ones(C))
    assert torch.allclose(z[0].cpu(), torch.full((C,), 1.25))   # 1 + (0.25-0.5)*(-1)
