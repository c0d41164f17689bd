"""Pins of the CPU fp64 oracle against facts that do not come from the oracle.

Each test checks a closed form, an invariant the definitions imply, a
hand-worked value (tests/golden/) or brute force on tiny inputs, chosen so
that a plausible slip in the oracle (dropped term, wrong sign, wrong index,
transposed operand, wrong pairing) fails at least one of them.  CPU only.
"""
import math
import os

import numpy as np
import pytest

import oracle as orc
from h3inputs import CONFIGS

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SECTIONS = (32, 48, 48)
OFFSETS = (0, 32, 80)


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


# ---------------------------------------------------------------- layout (a1)
def test_layout_counts_match_the_workloads():
    for line in _read_table("workloads.txt"):
        name, *vals = line.split()
        T, vt, vh, vw, ac, asteps, L = map(int, vals)
        cfg = CONFIGS[name]
        assert (cfg.n_text, cfg.video_t, cfg.video_h, cfg.video_w,
                cfg.audio_channels, cfg.audio_steps) == (T, vt, vh, vw, ac, asteps)
        mod, pos = orc.packed_layout(T, vt, vh, vw, ac, asteps)
        assert mod.shape == (L,) and pos.shape == (L, 3) and cfg.L == L
        assert np.count_nonzero(mod == orc.MOD_TEXT) == T
        assert np.count_nonzero(mod == orc.MOD_VIDEO) == vt * vh * vw
        assert np.count_nonzero(mod == orc.MOD_AUDIO) == ac * asteps
        # segments are contiguous, in the order text, video, audio
        assert np.all(np.diff(mod.astype(np.int64)) >= 0)


def test_full_size_geometry_from_the_pages():
    # 1440x1280 frames at 32x spatial downsampling; 10 s of audio at 40 Hz
    assert (1440 // 32, 1280 // 32) == (45, 40)
    assert 10 * 40 == 400
    assert 358 + 32 * 45 * 40 + 2 * 400 == 58758
    # the kernel-aligned length on the pages is 58,816 (+58 pad tokens): the
    # effective length leaves a ragged tail in 128-row tiles and in 64-row tiles
    assert 58816 - 58758 == 58 and 58816 % 64 == 0
    assert 58758 % 128 == 6 and 58758 % 64 == 6


def test_layout_positions_at_segment_boundaries():
    T, vt, vh, vw, ac, S = 5, 3, 4, 6, 2, 7
    mod, pos = orc.packed_layout(T, vt, vh, vw, ac, S)
    V = vt * vh * vw
    for i in range(T):
        assert mod[i] == 0 and tuple(pos[i]) == (i, i, i)
    assert mod[T] == 1 and tuple(pos[T]) == (0, 0, 0)
    assert tuple(pos[T + 1]) == (0, 0, 1)               # w is fastest
    assert tuple(pos[T + vw]) == (0, 1, 0)
    assert tuple(pos[T + vh * vw]) == (1, 0, 0)
    assert tuple(pos[T + V - 1]) == (vt - 1, vh - 1, vw - 1)
    assert mod[T + V] == 2 and tuple(pos[T + V]) == (0, 0, 0)
    assert tuple(pos[T + V + S - 1]) == (S - 1, 0, 0)   # channel 0, last step
    assert tuple(pos[T + V + S]) == (0, 0, 1)           # channel 1, step 0
    assert tuple(pos[-1]) == (S - 1, 0, 1)


# ------------------------------------------------------- LayerNorm (a2)
def test_layer_norm_hand_worked_rows():
    for line in _read_table("ln_exact.txt"):
        xs, ys = line.split("|")
        x = np.array([float(v) for v in xs.split()])[None, :]
        y = np.array([float(v) for v in ys.split()])[None, :]
        np.testing.assert_allclose(orc.layer_norm(x, 0.0), y, rtol=0, atol=1e-15)


def test_modulate_identity_and_variance_closed_form():
    rng = np.random.default_rng(0)
    L, d, eps = 7, 96, 1e-6
    x = rng.normal(1.5, 2.0, size=(L, d))
    mod = np.array([0, 1, 2, 0, 1, 2, 1], dtype=np.uint8)
    zero = np.zeros((3, d))
    y = orc.adaln_modulate(x, mod, zero, zero, eps)
    var = x.var(axis=1)
    np.testing.assert_allclose(y.mean(axis=1), 0.0, atol=1e-13)
    np.testing.assert_allclose((y ** 2).mean(axis=1), var / (var + eps), rtol=1e-12)
    # shift invariance of the normalisation
    np.testing.assert_allclose(orc.adaln_modulate(x + 3.25, mod, zero, zero, eps), y,
                               atol=1e-12)


def test_modulate_indexes_by_modality():
    rng = np.random.default_rng(1)
    L, d = 9, 64
    x = rng.normal(size=(L, d))
    mod = np.array([2, 0, 1, 1, 0, 2, 2, 0, 1], dtype=np.uint8)
    shift = np.stack([np.full(d, c) for c in (0.5, -1.25, 3.0)])
    scale = -np.ones((3, d))           # (1 + scale) = 0  ->  y = shift[mod]
    y = orc.adaln_modulate(x, mod, shift, scale, 1e-6)
    assert np.array_equal(y, shift[mod.astype(int)])
    # a pure scale: y = LN(x) * (1 + s_m), rows of each modality scale alike
    scale2 = np.stack([np.full(d, c) for c in (0.0, 1.0, -0.5)])
    y2 = orc.adaln_modulate(x, mod, np.zeros((3, d)), scale2, 1e-6)
    ln = orc.layer_norm(x, 1e-6)
    for n in range(L):
        np.testing.assert_allclose(y2[n], ln[n] * (1 + scale2[mod[n], 0]), atol=1e-14)


# ------------------------------------------------------- projections (a3, a6)
def test_linear_brute_force_and_orientation():
    rng = np.random.default_rng(2)
    a = rng.normal(size=(3, 5))
    w = rng.normal(size=(4, 5))        # [out, in]
    out = orc.linear(a, w)
    assert out.shape == (3, 4)
    for i in range(3):
        for j in range(4):
            ref = math.fsum(a[i, k] * w[j, k] for k in range(5))
            assert abs(out[i, j] - ref) < 1e-12
    # fused [I; I; I] projection copies its input into Q, K and V
    d = 6
    y = rng.normal(size=(4, d))
    eye3 = np.concatenate([np.eye(d)] * 3, axis=0)
    assert np.array_equal(orc.linear(y, eye3), np.concatenate([y, y, y], axis=1))


# ------------------------------------------------------- RoPE (a4)
def _rand_qkv(rng, L, H, dh=128, scale=1.0):
    return rng.normal(size=(L, 3 * H * dh)) * scale


def test_rope_preserves_norms_and_leaves_v():
    rng = np.random.default_rng(3)
    L, H, dh = 11, 3, 128
    qkv = _rand_qkv(rng, L, H)
    pos = rng.integers(0, 500, size=(L, 3)).astype(np.int32)
    r = orc.mrope(qkv, pos, H, dh)
    d = H * dh
    for blk in (0, 1):
        a = qkv[:, blk * d:(blk + 1) * d].reshape(L, H, dh)
        b = r[:, blk * d:(blk + 1) * d].reshape(L, H, dh)
        np.testing.assert_allclose(np.linalg.norm(b, axis=2), np.linalg.norm(a, axis=2),
                                   rtol=1e-13)
        # every (t|h|w) section keeps its own norm, too
        for o, n in zip(OFFSETS, SECTIONS):
            np.testing.assert_allclose(np.linalg.norm(b[..., o:o + n], axis=2),
                                       np.linalg.norm(a[..., o:o + n], axis=2), rtol=1e-13)
    assert np.array_equal(r[:, 2 * d:], qkv[:, 2 * d:])


def test_rope_zero_position_is_identity():
    rng = np.random.default_rng(4)
    qkv = _rand_qkv(rng, 4, 2)
    pos = np.zeros((4, 3), dtype=np.int32)
    assert np.array_equal(orc.mrope(qkv, pos, 2), qkv)


def test_rope_scores_depend_only_on_position_difference():
    rng = np.random.default_rng(5)
    L, H, dh = 6, 2, 128
    d = H * dh
    qkv = _rand_qkv(rng, L, H)
    pos = rng.integers(0, 60, size=(L, 3)).astype(np.int32)
    shift = np.array([[17, -5, 230]], dtype=np.int32)
    a = orc.mrope(qkv, pos, H)
    b = orc.mrope(qkv, pos + shift, H)
    for h in range(H):
        qa = a[:, h * dh:(h + 1) * dh]
        ka = a[:, d + h * dh:d + (h + 1) * dh]
        qb = b[:, h * dh:(h + 1) * dh]
        kb = b[:, d + h * dh:d + (h + 1) * dh]
        np.testing.assert_allclose(qb @ kb.T, qa @ ka.T, rtol=1e-9, atol=1e-9)
    # and a change of only one token's position does change its scores
    pos2 = pos.copy()
    pos2[0, 1] += 1
    c = orc.mrope(qkv, pos2, H)
    assert not np.allclose(c[:, :dh] @ c[:, d:d + dh].T, a[:, :dh] @ a[:, d:d + dh].T)


@pytest.mark.parametrize("axis", [0, 1, 2])
def test_rope_single_axis_rotation_closed_form(axis):
    """A unit vector on dim (o_a + 2j) turns inside the pair (o_a+2j, o_a+2j+1)
    by p * 10000**(-2j/n_a) when only axis ``axis`` has a nonzero position,
    and stays put when only another axis moves."""
    H, dh = 1, 128
    o, n = OFFSETS[axis], SECTIONS[axis]
    P = 7
    for j in (0, 1, n // 2 - 1):
        e = np.zeros((1, 3 * dh))
        e[0, o + 2 * j] = 1.0              # in Q
        e[0, dh + o + 2 * j + 1] = 1.0     # in K (the odd member of the pair)
        pos = np.zeros((1, 3), dtype=np.int32)
        pos[0, axis] = P
        r = orc.mrope(e, pos, H)
        phi = P * 10000.0 ** (-2.0 * j / n)
        want = np.zeros(3 * dh)
        want[o + 2 * j] = math.cos(phi)
        want[o + 2 * j + 1] = math.sin(phi)
        want[dh + o + 2 * j] = -math.sin(phi)
        want[dh + o + 2 * j + 1] = math.cos(phi)
        np.testing.assert_allclose(r[0], want, atol=1e-15)
        # moving a different axis leaves this section untouched
        pos_other = np.zeros((1, 3), dtype=np.int32)
        pos_other[0, (axis + 1) % 3] = P
        assert np.array_equal(orc.mrope(e, pos_other, H), e)


def test_rope_frequency_ladder_values():
    # t section: 16 pairs, ratio 10000**(-1/16) = 10**-0.25 between neighbours
    ang = orc.rope_angles(np.array([[1, 0, 0]], dtype=np.int32))
    assert ang.shape == (1, 64)
    assert ang[0, 0] == 1.0
    assert abs(ang[0, 1] - 10 ** -0.25) < 1e-15
    assert abs(ang[0, 15] - 10 ** (-0.25 * 15)) < 1e-15
    assert np.all(ang[0, 16:] == 0.0)
    # h section: 24 pairs, ratio 10000**(-1/24) = 10**(-1/6)
    ang = orc.rope_angles(np.array([[0, 1, 0]], dtype=np.int32))
    assert ang[0, 16] == 1.0 and abs(ang[0, 17] - 10 ** (-1 / 6)) < 1e-15
    assert np.all(ang[0, :16] == 0.0) and np.all(ang[0, 40:] == 0.0)


# ------------------------------------------------------- attention (a5)
def _pack(q, k, v):
    return np.concatenate([q, k, v], axis=1)


def test_attention_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(6)
    L, H, dh = 37, 2, 128
    q = rng.normal(size=(L, H * dh))
    k = np.tile(rng.normal(size=(1, H * dh)), (L, 1))
    v = rng.normal(size=(L, H * dh))
    o, lse = orc.attention(_pack(q, k, v), H, dh)
    np.testing.assert_allclose(o, np.tile(v.mean(axis=0), (L, 1)), atol=1e-13)
    # lse = s + log L for identical scores
    for h in range(H):
        s = (q[:, h * dh:(h + 1) * dh] @ k[0, h * dh:(h + 1) * dh]) / math.sqrt(dh)
        np.testing.assert_allclose(lse[h], s + math.log(L), atol=1e-12)


def test_attention_single_token_and_causal_first_row():
    rng = np.random.default_rng(7)
    H, dh = 2, 128
    qkv = rng.normal(size=(1, 3 * H * dh))
    o, _ = orc.attention(qkv, H, dh)
    assert np.allclose(o[0], qkv[0, 2 * H * dh:], atol=1e-15)
    qkv = rng.normal(size=(9, 3 * H * dh))
    o, _ = orc.attention(qkv, H, dh, causal=True)
    assert np.allclose(o[0], qkv[0, 2 * H * dh:], atol=1e-15)


def test_attention_brute_force_tiny():
    """Explicit per-score exp/sum loops (math.exp, math.fsum) on L <= 8."""
    rng = np.random.default_rng(8)
    H, dh = 2, 128
    d = H * dh
    for L, causal in ((5, False), (8, False), (8, True), (3, True)):
        qkv = rng.normal(size=(L, 3 * d)) * 1.7
        o, lse = orc.attention(qkv, H, dh, causal=causal)
        for h in range(H):
            for i in range(L):
                q = qkv[i, h * dh:(h + 1) * dh]
                keys = range(i + 1) if causal else range(L)
                s = {j: math.fsum(q[c] * qkv[j, d + h * dh + c] for c in range(dh))
                     / math.sqrt(dh) for j in keys}
                m = max(s.values())
                w = {j: math.exp(s[j] - m) for j in keys}
                z = math.fsum(w.values())
                for c in range(0, dh, 17):
                    ref = math.fsum(w[j] * qkv[j, 2 * d + h * dh + c] for j in keys) / z
                    assert abs(o[i, h * dh + c] - ref) < 1e-12
                assert abs(lse[h, i] - (m + math.log(z))) < 1e-12


def test_attention_invariances():
    rng = np.random.default_rng(9)
    L, H, dh = 23, 2, 128
    d = H * dh
    q, k, v = (rng.normal(size=(L, d)) for _ in range(3))
    o, lse = orc.attention(_pack(q, k, v), H, dh)
    # adding one vector u to every key shifts each score row by a constant
    u = rng.normal(size=(1, d))
    o2, lse2 = orc.attention(_pack(q, k + u, v), H, dh)
    np.testing.assert_allclose(o2, o, atol=1e-12)
    for h in range(H):
        du = (q[:, h * dh:(h + 1) * dh] @ u[0, h * dh:(h + 1) * dh]) / math.sqrt(dh)
        np.testing.assert_allclose(lse2[h], lse[h] + du, atol=1e-10)
    # permuting the keys together with their values changes nothing
    perm = rng.permutation(L)
    o3, _ = orc.attention(_pack(q, k[perm], v[perm]), H, dh)
    np.testing.assert_allclose(o3, o, atol=1e-12)
    # causal row i equals full attention over the prefix [0, i]
    oc, _ = orc.attention(_pack(q, k, v), H, dh, causal=True)
    for i in (0, 4, L - 1):
        op, _ = orc.attention(_pack(q[:i + 1], k[:i + 1], v[:i + 1]), H, dh,
                              rows=np.array([i]))
        np.testing.assert_allclose(oc[i], op[0], atol=1e-12)
    # a dominant key makes the softmax one-hot
    k4 = k.copy()
    k4[5] = q[2] * 50.0
    o4, _ = orc.attention(_pack(q, k4, v), H, dh, rows=np.array([2]))
    np.testing.assert_allclose(o4[0], v[5], atol=1e-9)
    # rows= selects the same numbers as the full call
    o5, _ = orc.attention(_pack(q, k, v), H, dh, rows=np.array([3, 11, 22]))
    np.testing.assert_allclose(o5, o[[3, 11, 22]], atol=1e-14)


# ------------------------------------------------------- gated residual (a6)
def test_gated_residual_special_cases():
    rng = np.random.default_rng(10)
    L, d = 6, 16
    x = rng.normal(size=(L, d))
    br = rng.normal(size=(L, d))
    mod = np.array([0, 1, 2, 2, 1, 0], dtype=np.uint8)
    assert np.array_equal(orc.gated_residual(x, br, mod, np.zeros((3, d))), x)
    gate = np.stack([np.full(d, c) for c in (0.25, -2.0, 8.0)])
    out = orc.gated_residual(np.zeros((L, d)), np.ones((L, d)), mod, gate)
    assert np.array_equal(out, gate[mod.astype(int)])


# ------------------------------------------------------- whole block (a7)
def test_block_special_weights_reduce_to_parts():
    rng = np.random.default_rng(11)
    cfg_T, vt, vh, vw, ac, S = 3, 1, 2, 2, 2, 2
    mod, pos = orc.packed_layout(cfg_T, vt, vh, vw, ac, S)
    L, H, dh = len(mod), 2, 128
    d = H * dh
    x = rng.normal(size=(L, d))
    shift, scale, gate = (rng.normal(size=(3, d)) * 0.1 for _ in range(3))
    wqkv = rng.normal(size=(3 * d, d)) / math.sqrt(d)
    wo = rng.normal(size=(d, d)) / math.sqrt(d)
    r = orc.block(x, mod, pos, shift, scale, gate, wqkv, wo, H)
    # gate = 0 -> out is x exactly
    r0 = orc.block(x, mod, pos, shift, scale, np.zeros((3, d)), wqkv, wo, H)
    assert np.array_equal(r0["out"], x)
    # Wo = 0 -> out is x exactly
    rz = orc.block(x, mod, pos, shift, scale, gate, wqkv, np.zeros((d, d)), H)
    assert np.array_equal(rz["out"], x)
    # composition of the parts
    y = orc.adaln_modulate(x, mod, shift, scale)
    np.testing.assert_allclose(r["y"], y, atol=0)
    np.testing.assert_allclose(r["qkv"], orc.mrope(y @ wqkv.T, pos, H), atol=1e-14)
    # the row-slice protocol gives the same rows as the full computation
    rows = np.array([0, 2, 5, L - 1])
    rs = orc.block_rows(x, mod, pos, shift, scale, gate, wqkv, wo, rows, H)
    for key in ("y", "O", "branch", "out"):
        np.testing.assert_allclose(rs[key], r[key][rows], atol=1e-12)
    np.testing.assert_allclose(rs["lse"], r["lse"][:, rows], atol=1e-12)
    for causal in (True,):
        rc = orc.block(x, mod, pos, shift, scale, gate, wqkv, wo, H, causal=causal)
        rcs = orc.block_rows(x, mod, pos, shift, scale, gate, wqkv, wo, rows, H,
                             causal=causal)
        np.testing.assert_allclose(rcs["out"], rc["out"][rows], atol=1e-12)


# ------------------------------------------------------- varlen attention (NEXT f1)
def test_varlen_visibility_matches_the_pages_example():
    """Brute force over exactly the keys the pages' example makes visible."""
    rng = np.random.default_rng(12)
    H, dh = 1, 128
    d = H * dh
    for line in _read_table("cu_seqlens_example.txt"):
        cu_s, q_s, lo_s, hi_s = line.split("|")
        cu = [int(v) for v in cu_s.split()]
        i, lo, hi = int(q_s), int(lo_s), int(hi_s)
        L = cu[-1]
        qkv = rng.normal(size=(L, 3 * d)) * 1.3
        o, _ = orc.attention_varlen(qkv, cu, H, dh, rows=np.array([i]))
        q = qkv[i, :d]
        s = {j: math.fsum(q[c] * qkv[j, d + c] for c in range(dh)) / math.sqrt(dh)
             for j in range(lo, hi + 1)}
        m = max(s.values())
        w = {j: math.exp(s[j] - m) for j in s}
        z = math.fsum(w.values())
        for c in range(0, dh, 9):
            ref = math.fsum(w[j] * qkv[j, 2 * d + c] for j in s) / z
            assert abs(o[0, c] - ref) < 1e-12
        # keys and values outside the visible range carry zero weight
        qkv2 = qkv.copy()
        outside = [j for j in range(L) if not lo <= j <= hi]
        qkv2[outside, d:] = rng.normal(size=(len(outside), 2 * d)) * 5
        o2, _ = orc.attention_varlen(qkv2, cu, H, dh, rows=np.array([i]))
        assert np.array_equal(o, o2)


def test_varlen_reduces_to_full_and_causal_within_segments():
    rng = np.random.default_rng(13)
    L, H, dh = 41, 2, 128
    qkv = rng.normal(size=(L, 3 * H * dh))
    full, lse_f = orc.attention(qkv, H, dh)
    one, lse_1 = orc.attention_varlen(qkv, [0, L], H, dh)
    assert np.array_equal(full, one) and np.array_equal(lse_f, lse_1)
    cu = [0, 7, 7, 30, 41]                     # an empty segment is allowed
    oc, _ = orc.attention_varlen(qkv, cu, H, dh, causal=True)
    for i, (lo, hi) in ((3, (0, 7)), (7, (7, 30)), (29, (7, 30)), (40, (30, 41))):
        op, _ = orc.attention(qkv[lo:i + 1], H, dh, rows=np.array([i - lo]))
        np.testing.assert_allclose(oc[i], op[0], atol=1e-12)


# ------------------------------------------------------- denoise step (NEXT f2)
def _straight_path(rng, L, C):
    x0 = rng.normal(size=(L, C))
    eps = rng.normal(size=(L, C))
    return x0, eps


def test_denoise_step_recovers_a_straight_path_exactly():
    """With the exact velocity of z = (1-s) x0 + s eps (H3 sign: x0 - eps), the
    clean estimate is x0 at any noise level and one Euler step lands on the
    path at the next level."""
    rng = np.random.default_rng(20)
    L, C = 12, 16
    mod = np.array([0, 1, 1, 2, 2, 1, 0, 2, 1, 1, 2, 2], dtype=np.uint8)
    x0, eps = _straight_path(rng, L, C)
    sig, sig_n = np.array([0.0, 0.8, 0.6]), np.array([0.0, 0.55, 0.2])
    s = sig[mod.astype(int)][:, None]
    sn = sig_n[mod.astype(int)][:, None]
    z = (1 - s) * x0 + s * eps
    z_next, x0_hat = orc.denoise_step(z, x0 - eps, mod, sig, sig_n, [0, 1, 1])
    lat = mod > 0
    np.testing.assert_allclose(x0_hat[lat], x0[lat], atol=1e-12)
    np.testing.assert_allclose(z_next[lat], ((1 - sn) * x0 + sn * eps)[lat], atol=1e-12)
    assert np.array_equal(z_next[~lat], z[~lat]) and np.array_equal(x0_hat[~lat], z[~lat])
    assert np.allclose(orc.sigma_to_t_h3([1.0, 0.25, 0.0]), [0.0, 0.75, 1.0])


def test_denoise_three_step_trace_reaches_clean_latents():
    sched = {}
    for line in _read_table("denoise_trace.txt"):
        name, vals = line.split("|")
        sched[name.strip()] = [float(v) for v in vals.split()]
    rng = np.random.default_rng(21)
    L, C = 10, 8
    mod = np.array([0, 1, 1, 1, 1, 2, 2, 2, 1, 2], dtype=np.uint8)
    anchor = np.zeros(L, dtype=np.uint8)
    anchor[[2, 6]] = 1
    x0, eps = _straight_path(rng, L, C)
    z_anchor = rng.normal(size=(L, C))
    z = eps.copy()                                     # pure noise at sigma_max = 1
    z[anchor.astype(bool)] = z_anchor[anchor.astype(bool)]
    for k in range(3):
        sig = [0.0, sched["video"][k], sched["audio"][k]]
        sig_n = [0.0, sched["video"][k + 1], sched["audio"][k + 1]]
        s = np.asarray(sig)[mod.astype(int)][:, None]
        v_h3 = x0 - eps                                # exact velocity, H3 sign
        z, x0_hat = orc.denoise_step(z, v_h3, mod, sig, sig_n, [0, 1, 1], anchor, z_anchor)
        a = anchor.astype(bool)
        assert np.array_equal(z[a], z_anchor[a])      # re-pinned every step
    free = (mod > 0) & ~anchor.astype(bool)
    np.testing.assert_allclose(z[free], x0[free], atol=1e-12)
    assert np.array_equal(z[mod == 0], eps[mod == 0])  # text rows never move


# ------------------------------------------------------- MLP sub-block (NEXT f3)
def test_gelu_identities_and_erf_form():
    u = np.linspace(-6, 6, 241)
    g = orc.gelu_tanh(u)
    # odd part: gelu(u) - gelu(-u) = u exactly for the 0.5 u (1 + t(u)) form with odd t
    np.testing.assert_allclose(g - orc.gelu_tanh(-u), u, atol=1e-13)
    # the tanh form stays within 1e-3 of the exact erf form u * Phi(u)
    exact = np.array([0.5 * v * (1 + math.erf(v / math.sqrt(2))) for v in u])
    assert np.max(np.abs(g - exact)) < 1e-3
    assert orc.gelu_tanh(np.array([0.0]))[0] == 0.0
    assert abs(orc.gelu_tanh(np.array([30.0]))[0] - 30.0) < 1e-12
    assert abs(orc.gelu_tanh(np.array([-30.0]))[0]) < 1e-12


def test_mlp_block_reductions():
    rng = np.random.default_rng(22)
    L, d, hid = 6, 16, 64
    x = rng.normal(size=(L, d))
    mod = np.array([0, 1, 2, 2, 1, 0], dtype=np.uint8)
    sh, sc, gt = (rng.normal(size=(3, d)) * 0.1 for _ in range(3))
    w1 = rng.normal(size=(hid, d)) / 4
    w2 = rng.normal(size=(d, hid)) / 8
    r = orc.mlp_block(x, mod, sh, sc, gt, w1, w2)
    assert np.array_equal(orc.mlp_block(x, mod, sh, sc, np.zeros((3, d)), w1, w2)["out"], x)
    assert np.array_equal(orc.mlp_block(x, mod, sh, sc, gt, w1, np.zeros((d, hid)))["out"], x)
    # brute-force one output element
    y = orc.adaln_modulate(x, mod, sh, sc)
    n, c = 3, 5
    hrow = [0.5 * u * (1 + math.tanh(math.sqrt(2 / math.pi) * (u + 0.044715 * u ** 3)))
            for u in (math.fsum(y[n, k] * w1[j, k] for k in range(d)) for j in range(hid))]
    ref = x[n, c] + gt[mod[n], c] * math.fsum(hrow[j] * w2[c, j] for j in range(hid))
    assert abs(r["out"][n, c] - ref) < 1e-12
