"""The seeded input generators (test infrastructure): geometry of the four
workloads, shapes, dtypes, distributions and determinism of both draws."""
import math

import torch

from h3inputs import CONFIGS, BlockConfig, block_inputs, block_inputs_device


def test_workload_geometry():
    # "Joint Audio-Video Generation in Production", §1: 58,758 effective tokens
    assert {k: c.L for k, c in CONFIGS.items()} == {
        "tiny": 64, "small": 4096, "medium": 16384, "full": 58758}
    full = CONFIGS["full"]
    assert (full.n_text, full.n_video, full.n_audio) == (358, 57600, 800)
    for c in CONFIGS.values():
        assert c.d == c.n_heads * c.head_dim and sum(c.rope_sections) == c.head_dim


def _check(inp, c, exact_seed_repeat):
    L, d, M = c.L, c.d, c.n_mod
    shapes = {"x": (L, d), "Wqkv": (3 * d, d), "Wo": (d, d), "shift": (M, d), "scale": (M, d),
              "gate": (M, d)}
    for k, shp in shapes.items():
        assert tuple(inp[k].shape) == shp, k
    for k in ("x", "Wqkv", "Wo"):
        assert inp[k].dtype == torch.bfloat16, k
    for k in ("shift", "scale", "gate"):
        assert inp[k].dtype == torch.float32, k
    std = {k: float(inp[k].float().std()) for k in shapes}
    assert abs(std["x"] - 1.0) < 0.02
    assert abs(std["Wqkv"] * math.sqrt(d) - 1.0) < 0.02
    assert abs(std["Wo"] * math.sqrt(d) - 1.0) < 0.02
    for k in ("shift", "scale", "gate"):
        assert abs(std[k] / 0.1 - 1.0) < 0.1
    for k in shapes:
        assert torch.equal(inp[k], exact_seed_repeat[k]), k


def test_block_inputs():
    c = CONFIGS["small"]
    _check(block_inputs(c), c, block_inputs(c))


def test_block_inputs_device_draw_on_the_cpu():
    c = BlockConfig("check", 16, 2, 8, 8, 2, 56, d=512, n_heads=4, seed=5)
    a = block_inputs_device(c, "cpu")
    _check(a, c, block_inputs_device(c, "cpu"))
    b = block_inputs_device(c, "cpu", seed=6)
    assert not torch.equal(a["x"], b["x"])
