"""The chain bound of the fused block's O and branch is a measurement.

Inside the fused block the attention output O and the branch O Wo^T inherit
the bf16 storage of y and of the rotated q, k, v.  This test builds that chain
with every step exact except the roundings the block's storage types force
(y, qkv and O stored in bf16, P rounded to bf16 before the P.V product), on 40
seeds of the tiny workload, and checks the two facts the GPU tests rely on:
the plain bound 2e-2 x RMS (+ 2^-8 |ref|) cannot hold for such a chain, and
the chain bound covers the worst chain with at least 25 % to spare.
"""
import math

import numpy as np
import torch

import oracle as orc
from h3inputs import CONFIGS, block_inputs
from tests._parity import BF16_U, CHAIN_MAX_REL_RMS, MAX_REL_RMS


def _bf16(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).double().numpy()


def _attention_p_rounded(qkv, H, dh=128):
    """softmax(q k^T / sqrt(dh)) v with the weights rounded to bf16 before
    they multiply v (the denominator keeps the unrounded weights)."""
    d = H * dh
    out = np.zeros((qkv.shape[0], d))
    for h in range(H):
        q = qkv[:, h * dh:(h + 1) * dh]
        k = qkv[:, d + h * dh:d + (h + 1) * dh]
        v = qkv[:, 2 * d + h * dh:2 * d + (h + 1) * dh]
        s = (q @ k.T) / math.sqrt(dh)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        out[:, h * dh:(h + 1) * dh] = (_bf16(p) @ v) / p.sum(axis=1, keepdims=True)
    return out


def _excess(got, ref):
    rms = np.sqrt(np.mean(ref * ref))
    return float((np.abs(got - ref) - BF16_U * np.abs(ref)).max() / rms)


def test_chain_bound_covers_an_exactly_rounded_chain():
    c = CONFIGS["tiny"]
    mod, pos = orc.packed_layout(c.n_text, c.video_t, c.video_h, c.video_w,
                                 c.audio_channels, c.audio_steps)
    worst_o = worst_b = 0.0
    for seed in range(40):
        inp = block_inputs(c, seed=seed)
        f = lambda k: inp[k].float().double().numpy()
        ref = orc.block(f("x"), mod, pos, f("shift"), f("scale"), f("gate"), f("Wqkv"),
                        f("Wo"), c.n_heads)
        y = _bf16(orc.adaln_modulate(f("x"), mod, f("shift"), f("scale")))
        qkv = _bf16(orc.mrope(orc.linear(y, f("Wqkv")), pos, c.n_heads))
        O = _bf16(_attention_p_rounded(qkv, c.n_heads))
        branch = _bf16(orc.linear(O, f("Wo")))
        worst_o = max(worst_o, _excess(O, ref["O"]))
        worst_b = max(worst_b, _excess(branch, ref["branch"]))
    worst = max(worst_o, worst_b)
    assert worst > MAX_REL_RMS, (worst_o, worst_b)
    assert 1.25 * worst <= CHAIN_MAX_REL_RMS, (worst_o, worst_b)
