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


_ORIG = {name: getattr(core, name) for name in
         ("layer_norm", "adaln_modulate", "linear", "rope_rotate_heads",
          "rope_angles", "attention", "attention_varlen", "gated_residual", "packed_layout",
          "denoise_step", "gelu_tanh")}

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
