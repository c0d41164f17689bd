"""Plant plausible mistakes in the oracle (CPU only) and check the pins catch them.

Each mutant replaces one oracle function with a subtly wrong variant; at
least one pin of tests/test_oracle_pins.py must then fail.
"""
import numpy as np
import pytest

import oracle
import oracle.h3_oracle as core
import tests.test_oracle_pins as pins


def _ln_unbiased(x, eps):
    mu = x.mean(axis=1, keepdims=True)
    var = ((x - mu) ** 2).sum(axis=1, keepdims=True) / (x.shape[1] - 1)
    return (x - mu) / np.sqrt(var + eps)


def _modulate_no_one(x, mod, shift, scale, eps=1e-6):
    m = mod.astype(np.int64)
    return core.layer_norm(x, eps) * scale[m] + shift[m]


def _linear_transposed(a, w):
    # reads the [out, in] weight buffer as if it were stored [in, out]
    return a @ w.reshape(w.shape[1], w.shape[0])


def _rotate_half_split(e, angles):
    h = e.shape[-1] // 2
    u, v = e[..., :h], e[..., h:]
    c = np.cos(angles)[:, None, :]
    s = np.sin(angles)[:, None, :]
    return np.concatenate([u * c - v * s, u * s + v * c], axis=-1)


def _rotate_sign_flipped(e, angles):
    return _ORIG["rope_rotate_heads"](e, -angles)


def _angles_shared_ladder(pos, sections=(32, 48, 48), base=10000.0):
    cols = []
    for a, n_a in enumerate(sections):
        j = np.arange(n_a // 2, dtype=np.float64)
        cols.append(pos[:, a:a + 1] * (base ** (-2.0 * j / 128))[None, :])
    return np.concatenate(cols, axis=1)


def _attention_no_scale(qkv, n_heads, head_dim=128, causal=False, sm_scale=None,
                        rows=None, k_rows_chunk=256):
    return _ORIG["attention"](qkv, n_heads, head_dim, causal, 1.0, rows, k_rows_chunk)


def _attention_causal_strict(qkv, n_heads, head_dim=128, causal=False, sm_scale=None,
                             rows=None, k_rows_chunk=256):
    """Off by one: under the causal mask a query does not see itself."""
    if not causal:
        return _ORIG["attention"](qkv, n_heads, head_dim, False, sm_scale, rows,
                                  k_rows_chunk)
    L = qkv.shape[0]
    d = n_heads * head_dim
    rows = np.arange(L) if rows is None else np.asarray(rows)
    out = np.zeros((len(rows), d))
    lse = np.zeros((n_heads, len(rows)))
    for r, i in enumerate(rows):
        keys = np.arange(max(int(i), 1))
        sub = np.concatenate([np.repeat(qkv[i:i + 1, :d], len(keys), 0),
                              qkv[keys, d:]], axis=1)
        o, l = _ORIG["attention"](sub, n_heads, head_dim, False, sm_scale,
                                  rows=np.array([0]))
        out[r], lse[:, r] = o[0], l[:, 0]
    return out, lse


def _varlen_boundary_off_by_one(qkv, cu_seqlens, n_heads, head_dim=128, causal=False,
                                sm_scale=None, rows=None):
    """A token on a segment start is put in the previous segment."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    L = qkv.shape[0]
    rows = np.arange(L) if rows is None else np.asarray(rows)
    d = n_heads * head_dim
    out = np.zeros((len(rows), d))
    lse = np.zeros((n_heads, len(rows)))
    seg = np.maximum(np.searchsorted(cu, rows, side="left") - 1, 0)
    for r, (i, s) in enumerate(zip(rows, seg)):
        lo, hi = int(cu[s]), int(cu[s + 1])
        if i >= hi:
            lo, hi = lo, i + 1
        o, l = _ORIG["attention"](qkv[lo:hi], n_heads, head_dim, causal, sm_scale,
                                  rows=np.array([i - lo]))
        out[r], lse[:, r] = o[0], l[:, 0]
    return out, lse


def _denoise_native_sign(z, v_h3, mod, sigma, sigma_next, update, anchor=None, z_anchor=None):
    """Uses H3's velocity without the sign reversal."""
    return _ORIG["denoise_step"](z, -v_h3, mod, sigma, sigma_next, update, anchor, z_anchor)


def _denoise_shared_schedule(z, v_h3, mod, sigma, sigma_next, update, anchor=None,
                             z_anchor=None):
    """Applies the video schedule to every modality."""
    s = np.full(len(sigma), sigma[1]); sn = np.full(len(sigma_next), sigma_next[1])
    return _ORIG["denoise_step"](z, v_h3, mod, s, sn, update, anchor, z_anchor)


def _gelu_sigmoid_form(u):
    """GELU by the sigmoid approximation u * sigmoid(1.702 u)."""
    return u / (1.0 + np.exp(-1.702 * u))


def _residual_wrong_index(x, branch, mod, gate):
    return x + gate[(mod.astype(np.int64) + 1) % 3] * branch


def _layout_audio_step_major(n_text, vt, vh, vw, ac, steps):
    mod, pos = _ORIG["packed_layout"](n_text, vt, vh, vw, ac, steps)
    T, V = n_text, vt * vh * vw
    k = 0
    for s in range(steps):
        for c in range(ac):
            pos[T + V + k] = (s, 0, c)
            k += 1
    return mod, pos


def _ln_eps_outside_sqrt(x, eps):
    mu = x.mean(axis=1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=1, keepdims=True)
    return (x - mu) / (np.sqrt(var) + eps)


def _modulate_shift_scale_swapped(x, mod, shift, scale, eps=1e-6):
    return _ORIG["adaln_modulate"](x, mod, scale, shift, eps)


def _angles_axes_swapped(pos, sections=(32, 48, 48), base=10000.0):
    """The h and w position columns exchanged."""
    return _ORIG["rope_angles"](np.asarray(pos)[:, [0, 2, 1]], sections, base)


def _mrope_rotates_v(qkv, pos, n_heads, head_dim=128, sections=(32, 48, 48), base=10000.0):
    out = _ORIG["mrope"](qkv, pos, n_heads, head_dim, sections, base)
    L, d = qkv.shape[0], n_heads * head_dim
    ang = core.rope_angles(pos, sections, base)
    out[:, 2 * d:] = core.rope_rotate_heads(qkv[:, 2 * d:].reshape(L, n_heads, head_dim),
                                            ang).reshape(L, d)
    return out


def _attention_v_from_k(qkv, n_heads, head_dim=128, causal=False, sm_scale=None, rows=None,
                        k_rows_chunk=256):
    """Values read from the K column block."""
    d = n_heads * head_dim
    swapped = qkv.copy()
    swapped[:, 2 * d:] = qkv[:, d:2 * d]
    return _ORIG["attention"](swapped, n_heads, head_dim, causal, sm_scale, rows, k_rows_chunk)


def _attention_head_mismatch(qkv, n_heads, head_dim=128, causal=False, sm_scale=None,
                             rows=None, k_rows_chunk=256):
    """Head h's queries meet the keys of head h + 1."""
    d = n_heads * head_dim
    moved = qkv.copy()
    moved[:, d:2 * d] = np.roll(qkv[:, d:2 * d], -head_dim, axis=1)
    return _ORIG["attention"](moved, n_heads, head_dim, causal, sm_scale, rows, k_rows_chunk)


def _block_residual_from_y(x, mod, pos, shift, scale, gate, wqkv, wo, n_heads, head_dim=128,
                           causal=False, eps=1e-6, sections=(32, 48, 48), base=10000.0,
                           cu_seqlens=None):
    """The residual taken from the modulated y instead of the block input x."""
    r = _ORIG["block"](x, mod, pos, shift, scale, gate, wqkv, wo, n_heads, head_dim, causal,
                       eps, sections, base, cu_seqlens)
    r["out"] = core.gated_residual(r["y"], r["branch"], mod, gate)
    return r


def _block_rows_k_unrotated(x, mod, pos, shift, scale, gate, wqkv, wo, rows, n_heads,
                            head_dim=128, causal=False, eps=1e-6, sections=(32, 48, 48),
                            base=10000.0):
    """The row-slice protocol forgets to rotate the keys of the other tokens."""
    d = n_heads * head_dim
    rows = np.asarray(rows, dtype=np.int64)
    y = core.adaln_modulate(x, mod, shift, scale, eps)
    kv = core.linear(y, wqkv[d:3 * d])
    q = core.rope_rotate_heads(core.linear(y[rows], wqkv[:d]).reshape(len(rows), n_heads,
                                                                       head_dim),
                               core.rope_angles(pos[rows], sections, base)).reshape(len(rows), d)
    qkv = np.zeros((x.shape[0], 3 * d))
    qkv[:, d:] = kv
    qkv[rows, :d] = q
    o, lse = core.attention(qkv, n_heads, head_dim, causal, rows=rows)
    branch = core.linear(o, wo)
    return {"y": y[rows], "q": q, "k": kv[:, :d], "v": kv[:, d:], "O": o, "lse": lse,
            "branch": branch, "out": core.gated_residual(x[rows], branch, mod[rows], gate)}


def _mlp_gelu_after_down(x, mod, shift, scale, gate, w1, w2, eps=1e-6):
    y = core.adaln_modulate(x, mod, shift, scale, eps)
    h = core.linear(y, w1)
    branch = core.gelu_tanh(core.linear(h, w2))
    return {"y": y, "h": h, "branch": branch,
            "out": core.gated_residual(x, branch, mod, gate)}


def _denoise_anchor_before_update(z, v_h3, mod, sigma, sigma_next, update, anchor=None,
                                  z_anchor=None):
    """Anchors restored before the update instead of after it."""
    z = np.array(z, dtype=np.float64, copy=True)
    if anchor is not None:
        a = np.asarray(anchor).astype(bool)
        z[a] = np.asarray(z_anchor)[a]
    return _ORIG["denoise_step"](z, v_h3, mod, sigma, sigma_next, update, None, None)


_ORIG = {name: getattr(core, name) for name in
         ("layer_norm", "adaln_modulate", "linear", "rope_rotate_heads",
          "rope_angles", "mrope", "attention", "attention_varlen", "gated_residual",
          "packed_layout", "block", "block_rows", "mlp_block", "denoise_step", "gelu_tanh")}

MUTANTS = {
    "unbiased-variance": ("layer_norm", _ln_unbiased),
    "modulate-without-one": ("adaln_modulate", _modulate_no_one),
    "transposed-weight": ("linear", _linear_transposed),
    "rope-half-split-pairs": ("rope_rotate_heads", _rotate_half_split),
    "rope-sign-flip": ("rope_rotate_heads", _rotate_sign_flipped),
    "rope-shared-ladder": ("rope_angles", _angles_shared_ladder),
    "attention-unscaled": ("attention", _attention_no_scale),
    "causal-excludes-self": ("attention", _attention_causal_strict),
    "gate-wrong-modality": ("gated_residual", _residual_wrong_index),
    "audio-step-major": ("packed_layout", _layout_audio_step_major),
    "varlen-boundary-off-by-one": ("attention_varlen", _varlen_boundary_off_by_one),
    "denoise-native-velocity-sign": ("denoise_step", _denoise_native_sign),
    "denoise-shared-schedule": ("denoise_step", _denoise_shared_schedule),
    "gelu-sigmoid-form": ("gelu_tanh", _gelu_sigmoid_form),
    "ln-eps-outside-sqrt": ("layer_norm", _ln_eps_outside_sqrt),
    "modulate-shift-scale-swapped": ("adaln_modulate", _modulate_shift_scale_swapped),
    "rope-h-w-positions-swapped": ("rope_angles", _angles_axes_swapped),
    "rope-rotates-v": ("mrope", _mrope_rotates_v),
    "attention-values-from-k-block": ("attention", _attention_v_from_k),
    "attention-keys-of-next-head": ("attention", _attention_head_mismatch),
    "block-residual-from-y": ("block", _block_residual_from_y),
    "block-rows-keys-unrotated": ("block_rows", _block_rows_k_unrotated),
    "mlp-gelu-after-down-projection": ("mlp_block", _mlp_gelu_after_down),
    "denoise-anchor-before-update": ("denoise_step", _denoise_anchor_before_update),
}

PIN_TESTS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_")]


def _run_pins():
    failed = []
    for t in PIN_TESTS:
        if hasattr(t, "pytestmark"):
            params = [m for m in t.pytestmark if m.name == "parametrize"]
            calls = [{params[0].args[0]: v} for v in params[0].args[1]] if params else [{}]
        else:
            calls = [{}]
        for kw in calls:
            try:
                t(**kw)
            except Exception:  # an assertion, or a crash caused by the mutant
                failed.append(t.__name__)
                break
    return failed


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_planted_mistake(mutant, monkeypatch):
    name, fn = MUTANTS[mutant]
    monkeypatch.setattr(core, name, fn)
    monkeypatch.setattr(oracle, name, fn)
    failed = _run_pins()
    assert failed, f"no pin caught the planted mistake {mutant!r}"


def test_unmutated_oracle_passes_all_pins():
    assert _run_pins() == []
