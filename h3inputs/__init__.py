"""Seeded synthetic inputs for the joint audio-video attention sub-block.

This module is shared by the oracle-side tests and the CUDA-side tests and
benchmark.  It holds the workload geometry and the random draws only: no
LayerNorm, projection, RoPE, attention or residual arithmetic lives here, and
it builds no per-token metadata (each side builds its own packed layout from
the segment counts below).

Workload geometry follows the pages' description of a MiniMax-H3 request:
one packed 1-D sequence of text, video and audio tokens (58,758 effective
tokens at full size; "Joint Audio-Video Generation in Production", §1 Unified
Architecture, pipeline table), video latents at 32x spatial / 4x temporal
compression and audio latents at 40 Hz per stereo channel ("DiffusionNFT on
MiniMax H3", section "MiniMax H3 and Why Joint Audio-Video Generation
Complicates RL Training").

Draw order for a block input set (CPU ``torch.Generator``): x, Wqkv, Wo,
shift, scale, gate.  x ~ N(0,1); weights ~ N(0, 1/d); modulation vectors
~ N(0, 0.1^2).  x and the weights are rounded to bf16 (both sides consume
the same bf16 values); shift/scale/gate stay fp32.
"""
from __future__ import annotations

import dataclasses
from typing import Dict

import torch

__all__ = ["BlockConfig", "CONFIGS", "block_inputs", "block_inputs_device", "sweep_modulation",
           "attention_qkv", "random_rows"]


@dataclasses.dataclass(frozen=True)
class BlockConfig:
    name: str
    n_text: int
    video_t: int
    video_h: int
    video_w: int
    audio_channels: int
    audio_steps: int
    d: int
    n_heads: int
    head_dim: int = 128
    seed: int = 0
    rope_sections: tuple = (32, 48, 48)
    rope_base: float = 10000.0
    ln_eps: float = 1e-6
    n_mod: int = 3

    @property
    def n_video(self) -> int:
        return self.video_t * self.video_h * self.video_w

    @property
    def n_audio(self) -> int:
        return self.audio_channels * self.audio_steps

    @property
    def L(self) -> int:
        return self.n_text + self.n_video + self.n_audio

    def flops(self, causal: bool = False) -> float:
        """Algorithmic FLOPs of one block forward (2 per multiply-add)."""
        L, d = self.L, self.d
        attn = 4.0 * d * (L * (L + 1) / 2.0 if causal else float(L) * L)
        return 6.0 * L * d * d + attn + 2.0 * L * d * d


CONFIGS: Dict[str, BlockConfig] = {
    # 64 = 16 text + 32 video (t2 h4 w4) + 16 audio (2 ch x 8 steps)
    "tiny": BlockConfig("tiny", 16, 2, 4, 4, 2, 8, d=256, n_heads=2, seed=0),
    # 4,096 = 256 + 3,584 (t7 h16 w32) + 256 (2 x 128)
    "small": BlockConfig("small", 256, 7, 16, 32, 2, 128, d=2048, n_heads=16, seed=1),
    # 16,384 = 384 + 15,360 (t12 h32 w40) + 640 (2 x 320: 8 s at 40 Hz)
    "medium": BlockConfig("medium", 384, 12, 32, 40, 2, 320, d=5120, n_heads=40, seed=2),
    # 58,758 = 358 + 57,600 (t32 h45 w40: 1440x1280 at 32x) + 800 (2 x 400: 10 s at 40 Hz)
    "full": BlockConfig("full", 358, 32, 45, 40, 2, 400, d=5120, n_heads=40, seed=3),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def block_inputs(cfg: BlockConfig, seed: int | None = None,
                 x_dtype: torch.dtype = torch.bfloat16) -> Dict[str, torch.Tensor]:
    """All inputs of one block forward, on the CPU.

    Returns bf16 ``x [L, d]``, ``Wqkv [3d, d]``, ``Wo [d, d]`` and fp32
    ``shift, scale, gate [n_mod, d]``.  ``x_raw`` holds the fp32 draw of x
    before rounding (the tiny case's fp32 I/O).
    """
    g = _gen(cfg.seed if seed is None else seed)
    L, d, M = cfg.L, cfg.d, cfg.n_mod
    std_w = 1.0 / (d ** 0.5)
    x_raw = torch.randn(L, d, generator=g, dtype=torch.float32)
    wqkv = torch.randn(3 * d, d, generator=g, dtype=torch.float32) * std_w
    wo = torch.randn(d, d, generator=g, dtype=torch.float32) * std_w
    shift = torch.randn(M, d, generator=g, dtype=torch.float32) * 0.1
    scale = torch.randn(M, d, generator=g, dtype=torch.float32) * 0.1
    gate = torch.randn(M, d, generator=g, dtype=torch.float32) * 0.1
    return {
        "x_raw": x_raw,
        "x": x_raw.to(x_dtype),
        "Wqkv": wqkv.to(torch.bfloat16),
        "Wo": wo.to(torch.bfloat16),
        "shift": shift,
        "scale": scale,
        "gate": gate,
    }


def block_inputs_device(cfg: BlockConfig, device, seed: int | None = None
                        ) -> Dict[str, torch.Tensor]:
    """The inputs of ``block_inputs`` (same names, shapes, dtypes and
    distributions, drawn in the same order) from a seeded ``torch.Generator``
    on ``device`` (torch's own Philox draw), for sequences long enough that a
    CPU draw of x (L*d values) takes minutes.  The tensors stay on ``device``;
    a test hands the oracle the rows it needs.  ``x_raw`` is omitted."""
    g = torch.Generator(device=device)
    g.manual_seed(int(cfg.seed if seed is None else seed))
    L, d, M = cfg.L, cfg.d, cfg.n_mod
    std_w = 1.0 / (d ** 0.5)

    def draw(*shape):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32)

    x = draw(L, d).to(torch.bfloat16)
    wqkv = (draw(3 * d, d) * std_w).to(torch.bfloat16)
    wo = (draw(d, d) * std_w).to(torch.bfloat16)
    mods = {k: draw(M, d) * 0.1 for k in ("shift", "scale", "gate")}
    return {"x": x, "Wqkv": wqkv, "Wo": wo, **mods}


def sweep_modulation(cfg: BlockConfig, step: int) -> Dict[str, torch.Tensor]:
    """Per-step modulation set of the denoising sweep (seed 1000 + step)."""
    g = _gen(1000 + int(step))
    M, d = cfg.n_mod, cfg.d
    return {k: torch.randn(M, d, generator=g, dtype=torch.float32) * 0.1
            for k in ("shift", "scale", "gate")}


def attention_qkv(L: int, n_heads: int, head_dim: int = 128, seed: int = 0,
                  qk_std: float = 1.0, v_std: float = 1.0) -> torch.Tensor:
    """A packed bf16 ``qkv [L, 3*H*dh]`` buffer ([Q | K | V], head-major).

    Used to exercise the attention call on its own.  ``qk_std`` controls how
    peaked the softmax is (scores have std ~ qk_std^2 after 1/sqrt(dh)).
    """
    g = _gen(seed)
    d = n_heads * head_dim
    q = torch.randn(L, d, generator=g) * qk_std
    k = torch.randn(L, d, generator=g) * qk_std
    v = torch.randn(L, d, generator=g) * v_std
    return torch.cat([q, k, v], dim=1).to(torch.bfloat16)


def random_rows(L: int, n: int, seed: int) -> torch.Tensor:
    """``n`` distinct sorted row indices in [0, L), always including 0 and L-1."""
    g = _gen(seed)
    n = min(n, L)
    perm = torch.randperm(L, generator=g)[:n]
    rows = torch.unique(torch.cat([perm, torch.tensor([0, L - 1])]))
    return rows.to(torch.int64)
