"""CPU fp64 oracle of one joint audio-video DiT attention sub-block.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline leg may import this module.  It shares no
code with the CUDA library and never imports it.

It computes the definition directly, in float64, with numpy: a matrix
product (BLAS) is the only library primitive used as a step; there is no
blocking, fusion, online softmax or reordering beyond the definition.  Every
function takes and returns numpy arrays; callers widen the bf16 inputs to
float64 before calling.

Sources (web pages describing MiniMax-H3 and its serving/training systems):
  [H3-RL]  "DiffusionNFT on MiniMax H3: Open-Source RL Training for Joint
           Audio-Video Generation" (gpts24.com), section "MiniMax H3 and Why
           Joint Audio-Video Generation Complicates RL Training".
  [vLLM]   "Joint Audio-Video Generation in Production: Architecture Deep Dive
           into MiniMax-H3 and vLLM-Omni", §1 Unified Architecture, §3 Packed
           Sequences and Modality Identity Preservation, §6 Boundary Trimming.
  [VeRL]   "多模态强化学习工程解析：VeRL-Omni 架构与 MiniMax-H3 训练实录",
           三 目标模型 (fused attention projections, shared AdaLN modulation).

Readings where the pages are silent (each is pinned by a CPU test):
  * modulate: y = LN(x) * (1 + scale[m]) + shift[m], LN without affine,
    biased variance, eps = 1e-6;
  * fused projection rows ordered [Q | K | V], head-major inside each block;
  * RoPE over (t, h, w): head dims [0,32) -> t, [32,80) -> h, [80,128) -> w,
    interleaved adjacent pairs (2j, 2j+1) inside each section, angle
    p_a * base^(-2j/n_a), same frequencies for every modality;
  * softmax scale 1/sqrt(head_dim); full bidirectional attention over the
    whole packed sequence, optional causal mask (key index <= query index);
  * out = x + gate[m] * (O Wo^T), residual is the pre-LN block input;
  * no biases, no padding: keys >= L do not exist.
Parity of the whole block is pinned only through the composition of the
pinned parts; the pages print no worked numeric example of the block.
"""
from __future__ import annotations

import math
from typing import Dict, Optional, Sequence, Tuple

import numpy as np

MOD_TEXT, MOD_VIDEO, MOD_AUDIO = 0, 1, 2


# ---------------------------------------------------------------------------
# a1: packed layout metadata  ([vLLM] §3, data-flow table and causal chain)
# ---------------------------------------------------------------------------
def packed_layout(n_text: int, video_t: int, video_h: int, video_w: int,
                  audio_channels: int, audio_steps: int
                  ) -> Tuple[np.ndarray, np.ndarray]:
    """Modality tag and (t, h, w) position of every token of the packed sequence.

    Order: text [0, T), then video row-major over (t, h, w), then audio
    channel-major (token T + V + c*S + s).  Positions: text (i, i, i), video
    (t, h, w), audio (step, 0, channel), all zero-based per modality.
    """
    mods = []
    pos = []
    for i in range(n_text):
        mods.append(MOD_TEXT)
        pos.append((i, i, i))
    for t in range(video_t):
        for h in range(video_h):
            for w in range(video_w):
                mods.append(MOD_VIDEO)
                pos.append((t, h, w))
    for c in range(audio_channels):
        for s in range(audio_steps):
            mods.append(MOD_AUDIO)
            pos.append((s, 0, c))
    return (np.asarray(mods, dtype=np.uint8),
            np.asarray(pos, dtype=np.int32).reshape(-1, 3))


# ---------------------------------------------------------------------------
# a2: modality-indexed AdaLN LayerNorm + modulate  ([H3-RL], AdaLN branches)
# ---------------------------------------------------------------------------
def layer_norm(x: np.ndarray, eps: float) -> np.ndarray:
    """Row-wise LayerNorm without affine: (x - mean) / sqrt(biased var + eps)."""
    mu = x.mean(axis=1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps)


def adaln_modulate(x: np.ndarray, mod: np.ndarray, shift: np.ndarray,
                   scale: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """y[n] = LN(x[n]) * (1 + scale[mod[n]]) + shift[mod[n]]."""
    m = mod.astype(np.int64)
    return layer_norm(x, eps) * (1.0 + scale[m]) + shift[m]


# ---------------------------------------------------------------------------
# a3 / a6: projections  ([VeRL] 三: fused QKV; nn.Linear layout W[out][in])
# ---------------------------------------------------------------------------
def linear(a: np.ndarray, w: np.ndarray) -> np.ndarray:
    """a @ w^T with w stored [out_features, in_features]; no bias."""
    return a @ w.T


# ---------------------------------------------------------------------------
# a4: 3D multimodal RoPE over (t, h, w)  ([H3-RL]; [vLLM] §3 tag + RoPE)
# ---------------------------------------------------------------------------
def rope_angles(pos: np.ndarray, sections: Sequence[int] = (32, 48, 48),
                base: float = 10000.0) -> np.ndarray:
    """Angle of every rotated pair: ``[L, head_dim/2]``.

    Pair k covers head dims (2k, 2k+1).  Section a (t, h, w) owns
    ``sections[a]`` consecutive dims; its j-th pair turns by
    ``pos[:, a] * base**(-2j / sections[a])``.
    """
    cols = []
    for a, n_a in enumerate(sections):
        j = np.arange(n_a // 2, dtype=np.float64)
        inv_freq = base ** (-2.0 * j / n_a)
        cols.append(pos[:, a:a + 1].astype(np.float64) * inv_freq[None, :])
    return np.concatenate(cols, axis=1)


def rope_rotate_heads(e: np.ndarray, angles: np.ndarray) -> np.ndarray:
    """Rotate ``e [L, H, dh]`` pairwise by ``angles [L, dh/2]`` (same for every head)."""
    u = e[..., 0::2]
    v = e[..., 1::2]
    c = np.cos(angles)[:, None, :]
    s = np.sin(angles)[:, None, :]
    out = np.empty_like(e)
    out[..., 0::2] = u * c - v * s
    out[..., 1::2] = u * s + v * c
    return out


def mrope(qkv: np.ndarray, pos: np.ndarray, n_heads: int, head_dim: int = 128,
          sections: Sequence[int] = (32, 48, 48), base: float = 10000.0
          ) -> np.ndarray:
    """Copy of ``qkv [L, 3*H*dh]`` with Q and K of every head rotated; V untouched."""
    assert sum(sections) == head_dim
    L = qkv.shape[0]
    d = n_heads * head_dim
    ang = rope_angles(pos, sections, base)
    out = qkv.copy()
    for blk in (0, 1):  # Q, K
        e = qkv[:, blk * d:(blk + 1) * d].reshape(L, n_heads, head_dim)
        out[:, blk * d:(blk + 1) * d] = rope_rotate_heads(e, ang).reshape(L, d)
    return out


# ---------------------------------------------------------------------------
# a5: joint attention over the whole packed sequence ([vLLM] §1 shared
#     attention context; §6: only the L effective tokens exist)
# ---------------------------------------------------------------------------
def attention(qkv: np.ndarray, n_heads: int, head_dim: int = 128,
              causal: bool = False, sm_scale: Optional[float] = None,
              rows: Optional[np.ndarray] = None, k_rows_chunk: int = 256
              ) -> Tuple[np.ndarray, np.ndarray]:
    """softmax(q k^T * sm_scale [+ causal mask]) v for every head.

    ``qkv`` is ``[L, 3*H*dh]``.  ``rows`` selects the query rows (default:
    all).  Returns ``O [R, H*dh]`` and the natural-log sum-exp ``lse [H, R]``
    of the scaled scores.  Two-pass softmax per query row: max, then
    exp/sum; a full score row is formed for every query.
    """
    L = qkv.shape[0]
    d = n_heads * head_dim
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(head_dim)
    if rows is None:
        rows = np.arange(L, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    R = rows.shape[0]
    out = np.zeros((R, d), dtype=np.float64)
    lse = np.zeros((n_heads, R), dtype=np.float64)
    keys = np.arange(L, dtype=np.int64)
    for h in range(n_heads):
        q = qkv[:, h * head_dim:(h + 1) * head_dim]
        k = qkv[:, d + h * head_dim:d + (h + 1) * head_dim]
        v = qkv[:, 2 * d + h * head_dim:2 * d + (h + 1) * head_dim]
        for r0 in range(0, R, k_rows_chunk):
            rr = rows[r0:r0 + k_rows_chunk]
            s = (q[rr] @ k.T) * sm_scale                      # [r, L]
            if causal:
                s = np.where(keys[None, :] <= rr[:, None], s, -np.inf)
            mx = s.max(axis=1, keepdims=True)
            p = np.exp(s - mx)
            den = p.sum(axis=1, keepdims=True)
            out[r0:r0 + len(rr), h * head_dim:(h + 1) * head_dim] = (p @ v) / den
            lse[h, r0:r0 + len(rr)] = (mx + np.log(den))[:, 0]
    return out, lse


def attention_varlen(qkv: np.ndarray, cu_seqlens, n_heads: int, head_dim: int = 128,
                     causal: bool = False, sm_scale: Optional[float] = None,
                     rows: Optional[np.ndarray] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Attention restricted to sub-sequences ([vLLM] §3, cu_seqlens and masks).

    ``cu_seqlens = [0, c1, ..., L]`` cuts the packed sequence into segments
    [c_s, c_{s+1}); a token attends only to keys of its own segment (and, when
    causal, to those at or before it).  This is attention applied to each
    segment's rows on their own.  Returns ``O [R, H*dh]`` and ``lse [H, R]``.
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    L = qkv.shape[0]
    assert cu[0] == 0 and cu[-1] == L and np.all(np.diff(cu) >= 0)
    if rows is None:
        rows = np.arange(L, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    d = n_heads * head_dim
    out = np.zeros((rows.shape[0], d), dtype=np.float64)
    lse = np.zeros((n_heads, rows.shape[0]), dtype=np.float64)
    seg = np.searchsorted(cu, rows, side="right") - 1
    for s in np.unique(seg):
        lo, hi = int(cu[s]), int(cu[s + 1])
        pick = np.nonzero(seg == s)[0]
        o, l = attention(qkv[lo:hi], n_heads, head_dim, causal, sm_scale, rows=rows[pick] - lo)
        out[pick] = o
        lse[:, pick] = l
    return out, lse


# ---------------------------------------------------------------------------
# a6: gated residual ([H3-RL] modality-specific AdaLN branches: the gate)
# ---------------------------------------------------------------------------
def gated_residual(x: np.ndarray, branch: np.ndarray, mod: np.ndarray,
                   gate: np.ndarray) -> np.ndarray:
    """out[n] = x[n] + gate[mod[n]] * branch[n]."""
    return x + gate[mod.astype(np.int64)] * branch


# ---------------------------------------------------------------------------
# a7: the whole sub-block
# ---------------------------------------------------------------------------
def block(x: np.ndarray, mod: np.ndarray, pos: np.ndarray, shift: np.ndarray,
          scale: np.ndarray, gate: np.ndarray, wqkv: np.ndarray, wo: np.ndarray,
          n_heads: int, head_dim: int = 128, causal: bool = False,
          eps: float = 1e-6, sections: Sequence[int] = (32, 48, 48),
          base: float = 10000.0, cu_seqlens=None) -> Dict[str, np.ndarray]:
    """Every intermediate of the block forward for all L tokens (attention
    restricted to the segments of ``cu_seqlens`` when given)."""
    y = adaln_modulate(x, mod, shift, scale, eps)
    qkv_pre = linear(y, wqkv)
    qkv = mrope(qkv_pre, pos, n_heads, head_dim, sections, base)
    if cu_seqlens is None:
        o, lse = attention(qkv, n_heads, head_dim, causal)
    else:
        o, lse = attention_varlen(qkv, cu_seqlens, n_heads, head_dim, causal)
    branch = linear(o, wo)
    out = gated_residual(x, branch, mod, gate)
    return {"y": y, "qkv_pre": qkv_pre, "qkv": qkv, "O": o, "lse": lse,
            "branch": branch, "out": out}


def block_rows(x: np.ndarray, mod: np.ndarray, pos: np.ndarray,
               shift: np.ndarray, scale: np.ndarray, gate: np.ndarray,
               wqkv: np.ndarray, wo: np.ndarray, rows: np.ndarray,
               n_heads: int, head_dim: int = 128, causal: bool = False,
               eps: float = 1e-6, sections: Sequence[int] = (32, 48, 48),
               base: float = 10000.0) -> Dict[str, np.ndarray]:
    """The block's outputs for the query rows ``rows`` only.

    Keys and values are formed for all L tokens (attention needs them); Q,
    O, the branch and out only for ``rows``.  Every number equals the
    corresponding row of :func:`block`.
    """
    d = n_heads * head_dim
    rows = np.asarray(rows, dtype=np.int64)
    y = adaln_modulate(x, mod, shift, scale, eps)
    kv_pre = linear(y, wqkv[d:3 * d])                            # [L, 2d]
    q_pre = linear(y[rows], wqkv[0:d])                           # [R, d]
    # rotate K (all tokens) and Q (selected rows) with their own positions
    L = x.shape[0]
    k_rot = rope_rotate_heads(kv_pre[:, :d].reshape(L, n_heads, head_dim),
                              rope_angles(pos, sections, base)).reshape(L, d)
    q_rot = rope_rotate_heads(q_pre.reshape(len(rows), n_heads, head_dim),
                              rope_angles(pos[rows], sections, base)
                              ).reshape(len(rows), d)
    qkv = np.empty((L, 3 * d), dtype=np.float64)
    qkv[:, d:2 * d] = k_rot
    qkv[:, 2 * d:] = kv_pre[:, d:]
    qkv[:, :d] = 0.0
    qkv[rows, :d] = q_rot
    o, lse = attention(qkv, n_heads, head_dim, causal, rows=rows)
    branch = linear(o, wo)
    out = gated_residual(x[rows], branch, mod[rows], gate)
    return {"y": y[rows], "q": q_rot, "k": k_rot, "v": kv_pre[:, d:],
            "O": o, "lse": lse, "branch": branch, "out": out}


# ---------------------------------------------------------------------------
# NEXT f2: one denoising-step update of the packed latent ([vLLM] §4
#   Denoising Execution Flow, stages 5-7; [VeRL] 5.1 timestep convention)
# ---------------------------------------------------------------------------
def sigma_to_t_h3(sigma):
    """H3's data-progress time for a noise level: t_H3 = 1 - sigma ([VeRL] 5.1)."""
    return 1.0 - np.asarray(sigma, dtype=np.float64)


def denoise_step(z: np.ndarray, v_h3: np.ndarray, mod: np.ndarray, sigma, sigma_next,
                 update, anchor: Optional[np.ndarray] = None,
                 z_anchor: Optional[np.ndarray] = None) -> Tuple[np.ndarray, np.ndarray]:
    """One deterministic (eta = 0) Euler step of the packed latent.

    ``z [L, C]`` is the state at noise level ``sigma[mod[n]]`` (one schedule per
    modality), ``v_h3 [L, C]`` the DiT's velocity in H3's sign (data-progress
    time), ``update[m]`` says whether modality m is a denoised latent (text
    rows are conditions and stay as they are).  With the straight path
    z = (1 - sigma) x0 + sigma eps the standard velocity is v = eps - x0 =
    -v_h3, the clean estimate is x0 = z - sigma v (rectified-flow v -> X0) and
    the Euler step to ``sigma_next`` is z + (sigma_next - sigma) v.  Rows with
    ``anchor[n]`` set are re-pinned to ``z_anchor[n]`` afterwards.
    Returns (z_next, x0_hat); rows that are not updated keep z in both.
    """
    m = mod.astype(np.int64)
    sig = np.asarray(sigma, dtype=np.float64)[m][:, None]
    sig_n = np.asarray(sigma_next, dtype=np.float64)[m][:, None]
    upd = np.asarray(update, dtype=bool)[m][:, None]
    v = -v_h3
    x0 = np.where(upd, z - sig * v, z)
    z_next = np.where(upd, z + (sig_n - sig) * v, z)
    if anchor is not None:
        a = np.asarray(anchor, dtype=bool)[:, None]
        z_next = np.where(a, z_anchor, z_next)
        x0 = np.where(a, z_anchor, x0)
    return z_next, x0


# ---------------------------------------------------------------------------
# NEXT f3: the MLP sub-block that completes one DiT layer ([H3-RL] "How
#   VeRL-Omni's Adapter Architecture Keeps H3-Specific Logic Contained": the
#   feed-forward projections ff.net.0.proj and ff.net.2; modality-specific
#   AdaLN branches).  Hidden width and activation are not given: 4d and the
#   tanh form of GELU are readings (parity of those choices unpinned).
# ---------------------------------------------------------------------------
def gelu_tanh(u: np.ndarray) -> np.ndarray:
    """GELU, tanh form: 0.5 u (1 + tanh(sqrt(2/pi) (u + 0.044715 u^3)))."""
    return 0.5 * u * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (u + 0.044715 * u ** 3)))


def mlp_block(x: np.ndarray, mod: np.ndarray, shift: np.ndarray, scale: np.ndarray,
              gate: np.ndarray, w1: np.ndarray, w2: np.ndarray, eps: float = 1e-6
              ) -> Dict[str, np.ndarray]:
    """out = x + gate[m] * (gelu(y W1^T) W2^T), y = LN(x)(1 + scale[m]) + shift[m].

    ``w1 [hidden, d]`` (ff.net.0.proj), ``w2 [d, hidden]`` (ff.net.2).
    """
    y = adaln_modulate(x, mod, shift, scale, eps)
    h = gelu_tanh(linear(y, w1))
    branch = linear(h, w2)
    return {"y": y, "h": h, "branch": branch, "out": gated_residual(x, branch, mod, gate)}

