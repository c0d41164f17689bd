"""The C-ABI library on a machine without a GPU: it builds, loads, exports
every entry point include/h3attn.h declares, rejects bad arguments before
launching anything, and its host-side packed layout equals the oracle's."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle as orc
from h3inputs import CONFIGS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from joint_audio_video_gb300 import build
    build.build()
    import joint_audio_video_gb300 as h3
    return h3


def _declared():
    with open(os.path.join(ROOT, "include", "h3attn.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const char\*|h3_status|void|int32_t)\s+(h3_\w+)\s*\(",
                                 text, re.M)))


def test_library_exports_every_declared_entry_point(lib):
    names = _declared()
    assert len(names) == 30, names
    raw = ctypes.CDLL(lib.lib_path)
    for n in names:
        assert hasattr(raw, n), f"{n} declared but not exported"
    assert sorted(lib.EXPORTED_SYMBOLS) == names
    assert lib.h3_version().startswith("h3attn")


def test_status_strings(lib):
    for code in range(7):
        assert lib.h3_status_string(code)
    assert lib.h3_status_string(99) == "unknown status"


def _bad(fn, *args):
    return fn(*args)


def test_invalid_arguments_are_rejected_before_any_launch(lib):
    L = lib.load()
    p = 1 << 20          # an aligned fake address: never dereferenced on these paths
    mis = p + 2          # misaligned
    INV, UNS = 1, 2
    # modulate: L < 1, d not a multiple of 128, null/misaligned pointers, n_mod range, eps
    assert L.h3_adaln_modulate(p, p, p, p, 0, 256, 3, 1e-6, p, None) == INV
    assert L.h3_adaln_modulate(p, p, p, p, 8, 200, 3, 1e-6, p, None) == INV
    assert L.h3_adaln_modulate(p, p, p, p, 8, 32768, 3, 1e-6, p, None) == INV
    assert L.h3_adaln_modulate(None, p, p, p, 8, 256, 3, 1e-6, p, None) == INV
    assert L.h3_adaln_modulate(mis, p, p, p, 8, 256, 3, 1e-6, p, None) == INV
    assert L.h3_adaln_modulate(p, p, p, p, 8, 256, 0, 1e-6, p, None) == INV
    assert L.h3_adaln_modulate(p, p, p, p, 8, 256, 256, 1e-6, p, None) == INV
    assert L.h3_adaln_modulate(p, p, p, p, 8, 256, 3, -1.0, p, None) == INV
    assert L.h3_adaln_modulate(p, p, p, p, 8, 256, 3, float("nan"), p, None) == INV
    # in-place y overlapping x partially
    assert L.h3_adaln_modulate(p, p, p, p, 8, 256, 3, 1e-6, p + 16, None) == INV
    # projection: overlap of y and qkv
    assert L.h3_qkv_proj(p, p, 8, 256, p, None) == INV
    assert L.h3_qkv_proj(p, p, 0, 256, p + (1 << 16), None) == INV
    # rope: head_dim, sections, base
    sec = (ctypes.c_int32 * 3)(32, 48, 48)
    bad_sec = (ctypes.c_int32 * 3)(32, 47, 49)
    short_sec = (ctypes.c_int32 * 3)(32, 48, 40)
    assert L.h3_mrope_apply(p, p, 8, 2, 64, ctypes.addressof(sec), 1e4, None) == UNS
    assert L.h3_mrope_apply(p, p, 8, 2, 128, ctypes.addressof(bad_sec), 1e4, None) == INV
    assert L.h3_mrope_apply(p, p, 8, 2, 128, ctypes.addressof(short_sec), 1e4, None) == INV
    assert L.h3_mrope_apply(p, p, 8, 2, 128, None, 1e4, None) == INV
    assert L.h3_mrope_apply(p, p, 8, 2, 128, ctypes.addressof(sec), -1.0, None) == INV
    # attention: head_dim, causal flag, scale, aliasing
    assert L.h3_joint_attn_fwd(p, 8, 2, 64, 0, 0.1, p + (1 << 16), None, None) == UNS
    assert L.h3_joint_attn_fwd(p, 8, 2, 128, 2, 0.1, p + (1 << 16), None, None) == INV
    assert L.h3_joint_attn_fwd(p, 8, 2, 128, 0, 0.0, p + (1 << 16), None, None) == INV
    assert L.h3_joint_attn_fwd(p, 8, 2, 128, 0, 0.1, p, None, None) == INV
    assert L.h3_joint_attn_fwd(p, 8, 2, 128, 0, 0.1, p + (1 << 16), mis, None) == INV
    # out projection: O aliasing out
    assert L.h3_out_proj_gated_residual(p, p, p + (1 << 16), p, p, 8, 256, 3, p, None) == INV
    assert L.h3_out_proj_gated_residual(p, p, p, p, p, 8, 256, 0, p + (1 << 16), None) == INV


def test_block_descriptor_and_workspace(lib):
    desc = lib.BlockDesc.make(L=58758, d=5120, n_heads=40)
    n = lib.h3_workspace_size(desc)
    L, d = 58758, 5120
    r = lambda x: (x + 255) // 256 * 256
    assert n == r(L * d * 2) + r(L * 3 * d * 2)
    for bad in (dict(L=0), dict(d=5000), dict(n_heads=39), dict(rope_sec=(32, 48, 50)),
                dict(ln_eps=-1.0), dict(n_mod=0), dict(rope_base=0.0)):
        kw = dict(L=64, d=256, n_heads=2)
        kw.update(bad)
        with pytest.raises(lib.H3Error) as e:
            lib.h3_workspace_size(lib.BlockDesc.make(**kw))
        assert e.value.status == 1
    with pytest.raises(lib.H3Error) as e:
        lib.h3_workspace_size(lib.BlockDesc.make(L=64, d=512, n_heads=8, head_dim=64))
    assert e.value.status == 2
    # a workspace that is too small is refused before launch
    desc = lib.BlockDesc.make(L=64, d=256, n_heads=2)
    need = lib.h3_workspace_size(desc)
    p = 1 << 24
    with pytest.raises(lib.H3Error) as e:
        lib.h3_attn_block_fwd(desc, p, p, p, p, p, p, p, p, 1 << 30, need - 1, p + (1 << 20),
                              stream=0)
    assert e.value.status == 6


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_host_layout_equals_oracle_bit_exact(lib, name):
    c = CONFIGS[name]
    args = (c.n_text, c.video_t, c.video_h, c.video_w, c.audio_channels, c.audio_steps)
    mod, pos = lib.h3_build_packed_layout(*args)
    omod, opos = orc.packed_layout(*args)
    assert mod.dtype == np.uint8 and pos.dtype == np.int32
    assert np.array_equal(mod, omod) and np.array_equal(pos, opos)


def test_host_layout_rejects_bad_counts(lib):
    with pytest.raises(lib.H3Error):
        lib.h3_build_packed_layout(0, 0, 0, 0, 0, 0)
    with pytest.raises(lib.H3Error):
        lib.h3_build_packed_layout(-1, 2, 2, 2, 2, 2)
    L = lib.load()
    mod = np.zeros(4, np.uint8)
    pos = np.zeros((4, 3), np.int32)
    assert L.h3_build_packed_layout(3, 1, 1, 2, 0, 0, mod.ctypes.data, pos.ctypes.data, 4) == 1


def test_segment_arrays_are_validated_before_launch(lib):
    L = lib.load()
    p = 1 << 20
    out = p + (1 << 24)
    import ctypes as C

    def call(cu, n_seg=None, Lt=45):
        arr = (C.c_int32 * len(cu))(*cu) if cu is not None else None
        n = len(cu) - 1 if n_seg is None else n_seg
        return L.h3_joint_attn_varlen_fwd(p, C.addressof(arr) if arr is not None else None, n, Lt,
                                          1, 128, 0, 0.088, out, None, None)
    assert call([1, 10, 45]) == 1            # does not start at 0
    assert call([0, 30, 10, 45]) == 1        # decreasing
    assert call([0, 10, 44]) == 1            # does not end at L
    assert call([0, 45], n_seg=0) == 1       # no segment
    assert call(None, n_seg=1) == 1          # NULL array
    assert call(list(range(0, 66)) + [45], Lt=45) == 1   # more than 64 segments
    with pytest.raises(lib.H3Error) as e:
        lib.h3_workspace_size(lib.BlockDesc.make(L=45, d=256, n_heads=2, cu_seqlens=[0, 10, 44]))
    assert e.value.status == 1
    assert lib.h3_workspace_size(lib.BlockDesc.make(L=45, d=256, n_heads=2,
                                                    cu_seqlens=[0, 10, 30, 45])) > 0


def test_denoise_arguments_are_validated_before_launch(lib):
    import ctypes as C
    L = lib.load()
    p = 1 << 20
    s3 = (C.c_float * 3)(0.0, 0.5, 0.5)
    bad = (C.c_float * 3)(0.0, 1.5, 0.5)
    up = (C.c_uint8 * 3)(0, 1, 1)
    a = lambda x: C.addressof(x)
    assert L.h3_denoise_step(p, None, p + (1 << 24), p, None, None, 10, 6, 3, a(s3), a(s3), a(up),
                             None) == 1                      # C not a multiple of 4
    assert L.h3_denoise_step(p, None, p + (1 << 24), p, None, None, 10, 8, 3, a(bad), a(s3), a(up),
                             None) == 1                      # sigma outside [0, 1]
    assert L.h3_denoise_step(p, None, p + (1 << 24), p, None, None, 10, 8, 3, None, a(s3), a(up),
                             None) == 1                      # missing host schedule
    assert L.h3_denoise_step(p + 4, None, p + (1 << 24), p, None, None, 10, 8, 3, a(s3), a(s3),
                             a(up), None) == 1               # misaligned state
    assert L.h3_denoise_step(p, p + 16, p + (1 << 24), p, None, None, 10, 8, 3, a(s3), a(s3),
                             a(up), None) == 1               # x0 overlapping z


def test_fp8_arguments_are_validated_before_launch(lib):
    L = lib.load()
    p = 1 << 20
    assert L.h3_quantize_rows_fp8(p, 4, 24, p + (1 << 24), p + (1 << 25), None) == 1   # K % 16
    assert L.h3_quantize_rows_fp8(p, 0, 32, p + (1 << 24), p + (1 << 25), None) == 1   # R < 1
    assert L.h3_gemm_fp8(p, p, p, p, 8, 200, 256, p, None) == 1      # N % 128
    assert L.h3_gemm_fp8(p, p, p, p, 8, 256, 64, p, None) == 1       # K % 128
    assert L.h3_gemm_fp8(p + 8, p, p, p, 8, 256, 256, p, None) == 1  # misaligned A
    desc = lib.BlockDesc.make(L=64, d=256, n_heads=2)
    assert lib.h3_workspace_size_fp8(desc) > lib.h3_workspace_size(desc)
    assert lib.h3_mlp_workspace_size_fp8(lib.MlpDesc.make(L=64, d=256)) > 0


def test_fp8_attention_arguments_are_validated_before_launch(lib):
    L = lib.load()
    p = 1 << 20
    r = lambda x: (x + 255) // 256 * 256
    # workspace: qk8 [L][2d] bytes | sq [H][L] fp32 | sk [H][ceil(L/128)] fp32
    for Lt, H in ((1, 1), (300, 2), (58758, 40)):
        assert lib.h3_attn_workspace_size_fp8(Lt, H) == (
            r(Lt * 2 * H * 128) + r(H * Lt * 4) + r(H * ((Lt + 127) // 128) * 4))
    n = ctypes.c_size_t(0)
    assert L.h3_attn_workspace_size_fp8(0, 2, 128, ctypes.byref(n)) == 1
    assert L.h3_attn_workspace_size_fp8(64, 2, 64, ctypes.byref(n)) == 2
    assert L.h3_attn_workspace_size_fp8(64, 2, 128, None) == 1
    big = 1 << 28
    # quantiser: alignment, null scales, head size, overlap with its input
    assert L.h3_quantize_qk_fp8(p + 8, 64, 2, 128, p + big, p + 2 * big, p + 3 * big, None) == 1
    assert L.h3_quantize_qk_fp8(p, 64, 2, 128, p + big, None, p + 3 * big, None) == 1
    assert L.h3_quantize_qk_fp8(p, 64, 2, 64, p + big, p + 2 * big, p + 3 * big, None) == 2
    assert L.h3_quantize_qk_fp8(p, 64, 2, 128, p + 4096, p + 2 * big, p + 3 * big, None) == 1
    assert L.h3_quantize_qk_fp8(p, 0, 2, 128, p + big, p + 2 * big, p + 3 * big, None) == 1
    # attention: workspace size and alignment, causal flag, scale, overlaps
    ws = lib.h3_attn_workspace_size_fp8(64, 2)
    args = lambda **k: (k.get("qkv", p), 64, 2, 128, k.get("causal", 0), k.get("scale", 0.0884),
                        k.get("ws", p + big), k.get("ws_bytes", ws), k.get("O", p + 2 * big),
                        k.get("lse", None), None)
    assert L.h3_joint_attn_fwd_fp8(*args(ws_bytes=ws - 1)) == 6
    assert L.h3_joint_attn_fwd_fp8(*args(ws=p + big + 16)) == 1
    assert L.h3_joint_attn_fwd_fp8(*args(causal=2)) == 1
    assert L.h3_joint_attn_fwd_fp8(*args(scale=0.0)) == 1
    assert L.h3_joint_attn_fwd_fp8(*args(scale=float("inf"))) == 1
    assert L.h3_joint_attn_fwd_fp8(*args(O=p + big + 256)) == 1      # O inside the workspace
    assert L.h3_joint_attn_fwd_fp8(*args(ws=p + 256)) == 1           # workspace over qkv
    assert L.h3_joint_attn_fwd_fp8(*args(lse=p + big + 4)) == 1      # lse inside the workspace
    assert L.h3_joint_attn_fwd_fp8(*args(O=p + 8)) == 1              # misaligned O
    # the fused fp8 block needs the score workspace only without segments
    d0 = lib.BlockDesc.make(L=64, d=256, n_heads=2)
    d1 = lib.BlockDesc.make(L=64, d=256, n_heads=2, cu_seqlens=[0, 20, 64])
    assert lib.h3_workspace_size_fp8(d0) - lib.h3_workspace_size_fp8(d1) == \
        lib.h3_attn_workspace_size_fp8(64, 2)


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    """No fallback: with the shared library absent, loading it and every call
    through the binding raise instead of computing anything elsewhere."""
    import pytest
    import torch

    import joint_audio_video_gb300 as h3

    monkeypatch.setattr(h3, "_lib", None)
    monkeypatch.setattr(h3, "lib_path", str(tmp_path / "libh3attn.so"))
    with pytest.raises(RuntimeError, match="is missing"):
        h3.load()
    x = torch.zeros(4, 128, dtype=torch.bfloat16)
    with pytest.raises(RuntimeError, match="is missing"):
        h3.h3_adaln_modulate(x, torch.zeros(4, dtype=torch.uint8), torch.zeros(1, 128),
                             torch.zeros(1, 128), 4, 128, 1, 1e-6, torch.empty_like(x))
    with pytest.raises(RuntimeError, match="is missing"):
        h3.h3_build_packed_layout(1, 1, 1, 1, 1, 1)


def test_extreme_counts_cannot_wrap_into_valid_sizes(lib):
    """A head count whose width n_heads * 128 wraps around 32 bits to a valid d,
    or an fp8 GEMM whose tile count would not fit 32 bits, is rejected before
    any launch."""
    L = lib.load()
    p = 1 << 20
    INV = 1
    wrap = (1 << 25) + 1            # (2^25 + 1) * 128 = 2^32 + 128 -> 128 in 32 bits
    sec = (ctypes.c_int32 * 3)(32, 48, 48)
    far = p + (1 << 30)
    assert L.h3_joint_attn_fwd(p, 8, wrap, 128, 0, 0.1, far, None, None) == INV
    assert L.h3_joint_attn_fwd(p, 8, 129, 128, 0, 0.1, far, None, None) == INV
    assert L.h3_mrope_apply(p, p, 8, wrap, 128, ctypes.addressof(sec), 1e4, None) == INV
    cu = (ctypes.c_int32 * 2)(0, 8)
    assert L.h3_joint_attn_varlen_fwd(p, ctypes.addressof(cu), 1, 8, wrap, 128, 0, 0.1, far,
                                      None, None) == INV
    desc = lib.BlockDesc.make(L=64, d=256, n_heads=2)
    desc.n_heads = wrap
    desc.d = 128                    # = wrap * 128 in 32 bits
    nbytes = ctypes.c_size_t(0)
    assert L.h3_workspace_size(ctypes.byref(desc), ctypes.byref(nbytes)) == INV
    big = (1 << 31) - 128
    assert L.h3_gemm_fp8(p, p, p, p, big, big, 128, far, None) == INV


def test_layout_counts_too_large_for_64_bits_are_rejected(lib):
    L = lib.load()
    big = (1 << 31) - 1
    mod = (ctypes.c_uint8 * 4)()
    pos = (ctypes.c_int32 * 12)()
    assert L.h3_build_packed_layout(0, big, big, big, 0, 0, mod, pos, 4) == 1
    assert L.h3_build_packed_layout(0, 0, 0, 0, big, big, mod, pos, 4) == 1
    assert L.h3_build_packed_layout(big, 1, 1, 1, 0, 0, mod, pos, 4) == 1
