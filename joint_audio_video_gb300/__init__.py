"""Python binding of libh3attn (the GB300 joint audio-video attention sub-block).

Argument marshalling only: every function below has the name of the C entry
point it calls, takes torch tensors (or raw integer addresses) and the
caller's CUDA stream, and raises :class:`H3Error` on a non-zero status.  All
arithmetic runs in the library's CUDA kernels; there is no other code path.
If the shared library is missing, :func:`load` raises instead of falling back.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import numpy as np

__all__ = [
    "H3Error", "BlockDesc", "load", "lib_path", "h3_version", "h3_status_string",
    "h3_build_packed_layout", "h3_adaln_modulate", "h3_qkv_proj", "h3_mrope_apply",
    "h3_joint_attn_fwd", "h3_joint_attn_varlen_fwd", "h3_out_proj_gated_residual",
    "h3_workspace_size",
    "h3_attn_block_fwd", "h3_sync_status", "h3_set_wait_limit_ns",
    "h3_selftest_wait_timeout", "h3_attn_block_fwd_profiled", "h3_attn_block_fwd_noalloc",
    "h3_denoise_step", "MlpDesc", "h3_mlp_workspace_size", "h3_mlp_block_fwd",
    "h3_quantize_rows_fp8", "h3_gemm_fp8", "h3_workspace_size_fp8", "h3_attn_block_fwd_fp8",
    "h3_mlp_workspace_size_fp8", "h3_mlp_block_fwd_fp8",
    "h3_attn_workspace_size_fp8", "h3_quantize_qk_fp8", "h3_joint_attn_fwd_fp8",
    "NOALLOC_SCRATCH_BYTES", "EXPORTED_SYMBOLS", "load_checked", "h3_checked_build",
    "h3_selftest_bounds_check",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_HERE, "libh3attn.so")
checked_lib_path = os.path.join(_HERE, "libh3attn_checked.so")

H3_OK = 0
STATUS_NAMES = {0: "H3_OK", 1: "H3_ERR_INVALID_ARG", 2: "H3_ERR_UNSUPPORTED", 3: "H3_ERR_CUDA",
                4: "H3_ERR_TIMEOUT", 5: "H3_ERR_BAD_INDEX", 6: "H3_ERR_WORKSPACE",
                7: "H3_ERR_OUT_OF_BOUNDS"}

EXPORTED_SYMBOLS = (
    "h3_status_string", "h3_version", "h3_build_packed_layout", "h3_adaln_modulate",
    "h3_qkv_proj", "h3_mrope_apply", "h3_joint_attn_fwd", "h3_joint_attn_varlen_fwd",
    "h3_out_proj_gated_residual",
    "h3_workspace_size", "h3_attn_block_fwd", "h3_sync_status", "h3_set_wait_limit_ns",
    "h3_selftest_wait_timeout", "h3_attn_block_fwd_profiled", "h3_attn_block_fwd_noalloc",
    "h3_denoise_step", "h3_mlp_workspace_size", "h3_mlp_block_fwd",
    "h3_quantize_rows_fp8", "h3_gemm_fp8", "h3_workspace_size_fp8", "h3_attn_block_fwd_fp8",
    "h3_mlp_workspace_size_fp8", "h3_mlp_block_fwd_fp8",
    "h3_attn_workspace_size_fp8", "h3_quantize_qk_fp8", "h3_joint_attn_fwd_fp8",
    "h3_checked_build", "h3_selftest_bounds_check",
)

# Workspace the library keeps per GPU for h3_attn_block_fwd_noalloc.
NOALLOC_SCRATCH_BYTES = 64 << 20


class H3Error(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)} ({msg})")
        self.status = status


class BlockDesc(ctypes.Structure):
    _fields_ = [("L", ctypes.c_int32), ("d", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("rope_sec", ctypes.c_int32 * 3),
                ("rope_base", ctypes.c_float), ("ln_eps", ctypes.c_float),
                ("causal", ctypes.c_int32), ("n_mod", ctypes.c_int32),
                ("n_seg", ctypes.c_int32), ("cu_seqlens", ctypes.POINTER(ctypes.c_int32))]

    @classmethod
    def make(cls, L, d, n_heads, head_dim=128, rope_sec=(32, 48, 48), rope_base=10000.0,
             ln_eps=1e-6, causal=False, n_mod=3, cu_seqlens=None) -> "BlockDesc":
        cu = None if cu_seqlens is None else _int32_array(cu_seqlens)
        desc = cls(int(L), int(d), int(n_heads), int(head_dim),
                   (ctypes.c_int32 * 3)(*[int(s) for s in rope_sec]), float(rope_base),
                   float(ln_eps), int(bool(causal)), int(n_mod),
                   0 if cu is None else len(cu) - 1, cu)
        desc._cu_keepalive = cu          # the struct points into this host array
        return desc


class MlpDesc(ctypes.Structure):
    _fields_ = [("L", ctypes.c_int32), ("d", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("ln_eps", ctypes.c_float), ("n_mod", ctypes.c_int32)]

    @classmethod
    def make(cls, L, d, hidden=None, ln_eps=1e-6, n_mod=3) -> "MlpDesc":
        return cls(int(L), int(d), int(4 * d if hidden is None else hidden), float(ln_eps),
                   int(n_mod))


def _int32_array(values):
    vals = [int(v) for v in values]
    return (ctypes.c_int32 * len(vals))(*vals)


_lib: Optional[ctypes.CDLL] = None
_P = ctypes.c_void_p
_I = ctypes.c_int32


def _sig(lib):
    lib.h3_status_string.restype = ctypes.c_char_p
    lib.h3_status_string.argtypes = [ctypes.c_int]
    lib.h3_version.restype = ctypes.c_char_p
    lib.h3_version.argtypes = []
    lib.h3_build_packed_layout.argtypes = [_I] * 6 + [_P, _P, ctypes.c_int64]
    lib.h3_adaln_modulate.argtypes = [_P, _P, _P, _P, _I, _I, _I, ctypes.c_float, _P, _P]
    lib.h3_qkv_proj.argtypes = [_P, _P, _I, _I, _P, _P]
    lib.h3_mrope_apply.argtypes = [_P, _P, _I, _I, _I, _P, ctypes.c_float, _P]
    lib.h3_joint_attn_fwd.argtypes = [_P, _I, _I, _I, _I, ctypes.c_float, _P, _P, _P]
    lib.h3_joint_attn_varlen_fwd.argtypes = [_P, _P, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P,
                                             _P]
    lib.h3_out_proj_gated_residual.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _P, _P]
    lib.h3_workspace_size.argtypes = [ctypes.POINTER(BlockDesc), ctypes.POINTER(ctypes.c_size_t)]
    lib.h3_attn_block_fwd.argtypes = [ctypes.POINTER(BlockDesc)] + [_P] * 9 + [ctypes.c_size_t,
                                                                                  _P, _P]
    lib.h3_attn_block_fwd_profiled.argtypes = (
        [ctypes.POINTER(BlockDesc)] + [_P] * 9 + [ctypes.c_size_t, _P, _P, _P])
    lib.h3_attn_block_fwd_noalloc.argtypes = [ctypes.POINTER(BlockDesc)] + [_P] * 10
    lib.h3_denoise_step.argtypes = [_P] * 6 + [_I, _I, _I, _P, _P, _P, _P]
    lib.h3_mlp_workspace_size.argtypes = [ctypes.POINTER(MlpDesc), ctypes.POINTER(ctypes.c_size_t)]
    lib.h3_mlp_block_fwd.argtypes = [ctypes.POINTER(MlpDesc)] + [_P] * 8 + [ctypes.c_size_t, _P,
                                                                            _P]
    lib.h3_quantize_rows_fp8.argtypes = [_P, _I, _I, _P, _P, _P]
    lib.h3_gemm_fp8.argtypes = [_P, _P, _P, _P, _I, _I, _I, _P, _P]
    lib.h3_workspace_size_fp8.argtypes = [ctypes.POINTER(BlockDesc), ctypes.POINTER(ctypes.c_size_t)]
    lib.h3_attn_block_fwd_fp8.argtypes = ([ctypes.POINTER(BlockDesc)] + [_P] * 11 +
                                          [ctypes.c_size_t, _P, _P])
    lib.h3_mlp_workspace_size_fp8.argtypes = [ctypes.POINTER(MlpDesc),
                                              ctypes.POINTER(ctypes.c_size_t)]
    lib.h3_mlp_block_fwd_fp8.argtypes = ([ctypes.POINTER(MlpDesc)] + [_P] * 10 +
                                         [ctypes.c_size_t, _P, _P])
    lib.h3_attn_workspace_size_fp8.argtypes = [_I, _I, _I, ctypes.POINTER(ctypes.c_size_t)]
    lib.h3_quantize_qk_fp8.argtypes = [_P, _I, _I, _I, _P, _P, _P, _P]
    lib.h3_joint_attn_fwd_fp8.argtypes = [_P, _I, _I, _I, _I, ctypes.c_float, _P,
                                          ctypes.c_size_t, _P, _P, _P]
    lib.h3_sync_status.argtypes = [_P]
    lib.h3_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.h3_set_wait_limit_ns.restype = None
    lib.h3_selftest_wait_timeout.argtypes = [ctypes.c_uint64, _P]
    lib.h3_checked_build.argtypes = []
    lib.h3_selftest_bounds_check.argtypes = [_P]
    for name in EXPORTED_SYMBOLS:
        if name not in ("h3_status_string", "h3_version", "h3_set_wait_limit_ns"):
            getattr(lib, name).restype = ctypes.c_int


def load() -> ctypes.CDLL:
    """Load libh3attn.so (built in-tree by ``build.build()``); raise if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(lib_path):
            raise RuntimeError(f"{lib_path} is missing: build it with "
                               "joint_audio_video_gb300.build.build() (needs nvcc)")
        lib = ctypes.CDLL(lib_path)
        _sig(lib)
        _lib = lib
    return _lib


def load_checked() -> ctypes.CDLL:
    """The checked library (libh3attn_checked.so, built in-tree by
    ``build.build(checked=True)``): the same entry points, every kernel's own
    global accesses bounds-tested (a failed test reports H3_ERR_OUT_OF_BOUNDS
    through h3_sync_status).  Loaded next to, not instead of, the library;
    call its entry points on the returned handle."""
    if not os.path.exists(checked_lib_path):
        raise RuntimeError(f"{checked_lib_path} is missing: build it with "
                           "joint_audio_video_gb300.build.build(checked=True) (needs nvcc)")
    lib = ctypes.CDLL(checked_lib_path)
    _sig(lib)
    return lib


def _addr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    raise TypeError(f"cannot take the address of {type(t)!r}")


def _stream(s) -> Optional[int]:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(fn: str, status: int) -> None:
    if status != H3_OK:
        raise H3Error(fn, status, load().h3_status_string(status).decode())


def h3_version() -> str:
    return load().h3_version().decode()


def h3_status_string(status: int) -> str:
    return load().h3_status_string(int(status)).decode()


def h3_build_packed_layout(n_text: int, video_t: int, video_h: int, video_w: int,
                           audio_channels: int, audio_steps: int):
    """Host layout: returns numpy ``mod [L] uint8`` and ``pos [L, 3] int32``."""
    L = n_text + video_t * video_h * video_w + audio_channels * audio_steps
    mod = np.zeros(max(L, 1), dtype=np.uint8)
    pos = np.zeros((max(L, 1), 3), dtype=np.int32)
    _check("h3_build_packed_layout", load().h3_build_packed_layout(
        n_text, video_t, video_h, video_w, audio_channels, audio_steps,
        mod.ctypes.data, pos.ctypes.data, L))
    return mod[:L], pos[:L]


def h3_adaln_modulate(x, mod, shift, scale, L, d, n_mod, eps, y, stream=None) -> None:
    _check("h3_adaln_modulate", load().h3_adaln_modulate(
        _addr(x), _addr(mod), _addr(shift), _addr(scale), L, d, n_mod, eps, _addr(y),
        _stream(stream)))


def h3_qkv_proj(y, Wqkv, L, d, qkv, stream=None) -> None:
    _check("h3_qkv_proj", load().h3_qkv_proj(_addr(y), _addr(Wqkv), L, d, _addr(qkv),
                                             _stream(stream)))


def h3_mrope_apply(qkv, pos, L, n_heads, head_dim=128, sec=(32, 48, 48), base=10000.0,
                   stream=None) -> None:
    sec_arr = (ctypes.c_int32 * 3)(*[int(s) for s in sec])
    _check("h3_mrope_apply", load().h3_mrope_apply(
        _addr(qkv), _addr(pos), L, n_heads, head_dim, ctypes.addressof(sec_arr), base,
        _stream(stream)))


def h3_joint_attn_fwd(qkv, L, n_heads, head_dim, causal, sm_scale, O, lse=None,
                      stream=None) -> None:
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(head_dim)
    _check("h3_joint_attn_fwd", load().h3_joint_attn_fwd(
        _addr(qkv), L, n_heads, head_dim, int(bool(causal)), sm_scale, _addr(O), _addr(lse),
        _stream(stream)))


def h3_joint_attn_varlen_fwd(qkv, cu_seqlens, L, n_heads, head_dim, causal, sm_scale, O,
                             lse=None, stream=None) -> None:
    """``cu_seqlens``: host sequence [0, c1, ..., L] of segment offsets."""
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(head_dim)
    cu = _int32_array(cu_seqlens)
    _check("h3_joint_attn_varlen_fwd", load().h3_joint_attn_varlen_fwd(
        _addr(qkv), ctypes.addressof(cu), len(cu) - 1, L, n_heads, head_dim, int(bool(causal)),
        sm_scale, _addr(O), _addr(lse), _stream(stream)))


def h3_out_proj_gated_residual(O, Wo, x_res, mod, gate, L, d, n_mod, out, stream=None) -> None:
    _check("h3_out_proj_gated_residual", load().h3_out_proj_gated_residual(
        _addr(O), _addr(Wo), _addr(x_res), _addr(mod), _addr(gate), L, d, n_mod, _addr(out),
        _stream(stream)))


def h3_workspace_size(desc: BlockDesc) -> int:
    n = ctypes.c_size_t(0)
    _check("h3_workspace_size", load().h3_workspace_size(ctypes.byref(desc), ctypes.byref(n)))
    return int(n.value)


def h3_attn_block_fwd(desc: BlockDesc, x, mod, pos, shift, scale, gate, Wqkv, Wo, workspace,
                      workspace_bytes, out, stream=None) -> None:
    _check("h3_attn_block_fwd", load().h3_attn_block_fwd(
        ctypes.byref(desc), _addr(x), _addr(mod), _addr(pos), _addr(shift), _addr(scale),
        _addr(gate), _addr(Wqkv), _addr(Wo), _addr(workspace), int(workspace_bytes), _addr(out),
        _stream(stream)))


def h3_attn_block_fwd_profiled(desc: BlockDesc, x, mod, pos, shift, scale, gate, Wqkv, Wo,
                               workspace, workspace_bytes, out, events, stream=None) -> None:
    """``events``: five ``torch.cuda.Event`` (or raw cudaEvent_t handles) or None."""
    arr = None
    if events is not None:
        handles = []
        for e in events:
            if not isinstance(e, int) and e.cuda_event == 0:
                # torch creates the CUDA event on its first record
                e.record(None if stream is None or isinstance(stream, int) else stream)
            handles.append(e if isinstance(e, int) else e.cuda_event)
        assert len(handles) == 5
        arr = (ctypes.c_void_p * 5)(*handles)
    _check("h3_attn_block_fwd_profiled", load().h3_attn_block_fwd_profiled(
        ctypes.byref(desc), _addr(x), _addr(mod), _addr(pos), _addr(shift), _addr(scale),
        _addr(gate), _addr(Wqkv), _addr(Wo), _addr(workspace), int(workspace_bytes), _addr(out),
        _stream(stream), arr))


def h3_attn_block_fwd_noalloc(desc: BlockDesc, x, mod, pos, shift, scale, gate, Wqkv, Wo, out,
                              stream=None) -> None:
    """The fused block on the library's own per-GPU workspace (no allocation
    anywhere); for shapes whose workspace fits NOALLOC_SCRATCH_BYTES."""
    _check("h3_attn_block_fwd_noalloc", load().h3_attn_block_fwd_noalloc(
        ctypes.byref(desc), _addr(x), _addr(mod), _addr(pos), _addr(shift), _addr(scale),
        _addr(gate), _addr(Wqkv), _addr(Wo), _addr(out), _stream(stream)))


def h3_denoise_step(z, x0, v_h3, mod, anchor, z_anchor, L, C, sigma, sigma_next, update,
                    stream=None) -> None:
    """``sigma``, ``sigma_next``, ``update``: host sequences, one entry per modality."""
    n_mod = len(sigma)
    sg = (ctypes.c_float * n_mod)(*[float(v) for v in sigma])
    sn = (ctypes.c_float * n_mod)(*[float(v) for v in sigma_next])
    up = (ctypes.c_uint8 * n_mod)(*[1 if u else 0 for u in update])
    _check("h3_denoise_step", load().h3_denoise_step(
        _addr(z), _addr(x0), _addr(v_h3), _addr(mod), _addr(anchor), _addr(z_anchor), L, C,
        n_mod, ctypes.addressof(sg), ctypes.addressof(sn), ctypes.addressof(up),
        _stream(stream)))


def h3_mlp_workspace_size(desc: MlpDesc) -> int:
    n = ctypes.c_size_t(0)
    _check("h3_mlp_workspace_size",
           load().h3_mlp_workspace_size(ctypes.byref(desc), ctypes.byref(n)))
    return int(n.value)


def h3_mlp_block_fwd(desc: MlpDesc, x, mod, shift, scale, gate, W1, W2, workspace,
                     workspace_bytes, out, stream=None) -> None:
    _check("h3_mlp_block_fwd", load().h3_mlp_block_fwd(
        ctypes.byref(desc), _addr(x), _addr(mod), _addr(shift), _addr(scale), _addr(gate),
        _addr(W1), _addr(W2), _addr(workspace), int(workspace_bytes), _addr(out),
        _stream(stream)))


def h3_quantize_rows_fp8(x, R, K, q, scale, stream=None) -> None:
    _check("h3_quantize_rows_fp8", load().h3_quantize_rows_fp8(
        _addr(x), R, K, _addr(q), _addr(scale), _stream(stream)))


def h3_gemm_fp8(A, a_scale, B, b_scale, M, N, K, C, stream=None) -> None:
    _check("h3_gemm_fp8", load().h3_gemm_fp8(_addr(A), _addr(a_scale), _addr(B), _addr(b_scale),
                                             M, N, K, _addr(C), _stream(stream)))


def h3_attn_workspace_size_fp8(L, n_heads, head_dim=128) -> int:
    n = ctypes.c_size_t(0)
    _check("h3_attn_workspace_size_fp8",
           load().h3_attn_workspace_size_fp8(L, n_heads, head_dim, ctypes.byref(n)))
    return int(n.value)


def h3_quantize_qk_fp8(qkv, L, n_heads, head_dim, qk8, sq, sk, stream=None) -> None:
    _check("h3_quantize_qk_fp8", load().h3_quantize_qk_fp8(
        _addr(qkv), L, n_heads, head_dim, _addr(qk8), _addr(sq), _addr(sk), _stream(stream)))


def h3_joint_attn_fwd_fp8(qkv, L, n_heads, head_dim, causal, sm_scale, workspace,
                          workspace_bytes, O, lse=None, stream=None) -> None:
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(head_dim)
    _check("h3_joint_attn_fwd_fp8", load().h3_joint_attn_fwd_fp8(
        _addr(qkv), L, n_heads, head_dim, int(bool(causal)), sm_scale, _addr(workspace),
        int(workspace_bytes), _addr(O), _addr(lse), _stream(stream)))


def h3_workspace_size_fp8(desc: BlockDesc) -> int:
    n = ctypes.c_size_t(0)
    _check("h3_workspace_size_fp8",
           load().h3_workspace_size_fp8(ctypes.byref(desc), ctypes.byref(n)))
    return int(n.value)


def h3_attn_block_fwd_fp8(desc: BlockDesc, x, mod, pos, shift, scale, gate, Wqkv_q, Wqkv_s,
                          Wo_q, Wo_s, workspace, workspace_bytes, out, stream=None) -> None:
    _check("h3_attn_block_fwd_fp8", load().h3_attn_block_fwd_fp8(
        ctypes.byref(desc), _addr(x), _addr(mod), _addr(pos), _addr(shift), _addr(scale),
        _addr(gate), _addr(Wqkv_q), _addr(Wqkv_s), _addr(Wo_q), _addr(Wo_s), _addr(workspace),
        int(workspace_bytes), _addr(out), _stream(stream)))


def h3_mlp_workspace_size_fp8(desc: MlpDesc) -> int:
    n = ctypes.c_size_t(0)
    _check("h3_mlp_workspace_size_fp8",
           load().h3_mlp_workspace_size_fp8(ctypes.byref(desc), ctypes.byref(n)))
    return int(n.value)


def h3_mlp_block_fwd_fp8(desc: MlpDesc, x, mod, shift, scale, gate, W1_q, W1_s, W2_q, W2_s,
                         workspace, workspace_bytes, out, stream=None) -> None:
    _check("h3_mlp_block_fwd_fp8", load().h3_mlp_block_fwd_fp8(
        ctypes.byref(desc), _addr(x), _addr(mod), _addr(shift), _addr(scale), _addr(gate),
        _addr(W1_q), _addr(W1_s), _addr(W2_q), _addr(W2_s), _addr(workspace),
        int(workspace_bytes), _addr(out), _stream(stream)))


def h3_sync_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status as a code."""
    return int(load().h3_sync_status(_stream(stream)))


def h3_set_wait_limit_ns(limit_ns: int) -> None:
    load().h3_set_wait_limit_ns(int(limit_ns))


def h3_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    _check("h3_selftest_wait_timeout",
           load().h3_selftest_wait_timeout(int(limit_ns), _stream(stream)))


def h3_checked_build() -> bool:
    return bool(load().h3_checked_build())


def h3_selftest_bounds_check(stream=None) -> int:
    """Returns the entry point's status: H3_ERR_UNSUPPORTED (2) in the normal
    build, which launches nothing; in the checked build, after the launch, the
    next h3_sync_status() reports H3_ERR_OUT_OF_BOUNDS."""
    return int(load().h3_selftest_bounds_check(_stream(stream)))
