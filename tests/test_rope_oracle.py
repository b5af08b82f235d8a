"""Rotary position embedding and QK-norm in the oracle (Qwen3-style backbones, X-MoD
notes "backbone configuration"; the NEXT row "RoPE at original positions, QK-norm"),
pinned to properties the transforms have by construction:
  * the rotation keeps each head vector's length and is the identity at position 0;
  * rotated q . k depends only on the position difference, so a block whose every
    position shifts by a constant is unchanged;
  * QK-norm leaves each head vector with unit RMS (gain 1) and makes the block blind to
    the scale of Wq and Wk;
  * a sparse layer rotates at the tokens' original positions: selecting every other
    token differs from selecting a prefix of the same tokens (which compact positions
    could not tell apart)."""
import math

import numpy as np

import oracle as O
from sparse_depth_token_gb300 import inputs as I

THETA = 1e4


def test_rotation_keeps_length_and_fixes_position_zero():
    g = np.random.default_rng(1)
    heads, hd = 3, 32
    x = g.standard_normal((5, heads * hd))
    y = O.qk_transform(x, heads, hd, theta=THETA, pos=np.array([0, 1, 7, 100, 4095]))
    nx = np.linalg.norm(x.reshape(5, heads, hd), axis=2)
    ny = np.linalg.norm(y.reshape(5, heads, hd), axis=2)
    np.testing.assert_allclose(ny, nx, rtol=1e-13)
    np.testing.assert_array_equal(y[0], x[0])
    assert np.abs(y[1:] - x[1:]).max() > 1e-3


def test_rotated_dot_product_depends_on_the_offset_only():
    g = np.random.default_rng(2)
    hd = 64
    q, k = g.standard_normal((1, hd)), g.standard_normal((1, hd))
    for p1, p2, c in ((9, 3, 11), (0, 40, 1000), (77, 77, 5)):
        a = O.qk_transform(q, 1, hd, theta=THETA, pos=[p1]) @ O.qk_transform(k, 1, hd, theta=THETA, pos=[p2]).T
        b = O.qk_transform(q, 1, hd, theta=THETA, pos=[p1 + c]) @ O.qk_transform(k, 1, hd, theta=THETA, pos=[p2 + c]).T
        np.testing.assert_allclose(a, b, rtol=1e-9)


def test_rotation_angles_and_pairing_closed_form():
    """The rotary embedding's definition evaluated by hand (rotate-half convention of the
    Qwen / LLaMA family): dimension c pairs with c + hd/2 and turns by t·θ^(−2c/hd).
    hd = 4, θ = 16, t = 3: pair (0, 2) turns by 3 rad, pair (1, 3) by 3·16^(−1/2) = 0.75
    rad. Basis vectors come out as the columns of the two plane rotations. An exponent of
    −c/hd (1.5 rad on the second pair) or interleaved pairs (0, 1), (2, 3) fail."""
    hd, theta, t = 4, 16.0, 3
    y = O.qk_transform(np.eye(hd), 1, hd, theta=theta, pos=[t] * hd)
    c0, s0 = math.cos(3.0), math.sin(3.0)
    c1, s1 = math.cos(0.75), math.sin(0.75)
    want = np.array([[c0, 0.0, s0, 0.0],      # e_0 -> (cos, sin) in the plane (0, 2)
                     [0.0, c1, 0.0, s1],      # e_1 -> (cos, sin) in the plane (1, 3)
                     [-s0, 0.0, c0, 0.0],     # e_2 -> (-sin, cos) in the plane (0, 2)
                     [0.0, -s1, 0.0, c1]])    # e_3 -> (-sin, cos) in the plane (1, 3)
    np.testing.assert_allclose(y, want, rtol=0, atol=1e-15)


def _layer(w, g_scale=1.0, wqk_scale=1.0, theta=THETA):
    lw = I.layer_weights(w, 6)
    g = np.random.default_rng(3)
    lw = dict(lw, wq=lw["wq"] * wqk_scale, wk=lw["wk"] * wqk_scale,
              gq=g_scale * (1 + 0.1 * g.standard_normal(w.hd)),
              gk=g_scale * (1 + 0.1 * g.standard_normal(w.hd)), rope_theta=theta)
    return lw


def test_block_is_unchanged_by_a_common_position_shift():
    w = I.WORKLOADS["tiny_fp32"]
    od = O.dims(w.B, w.T, w.d, w.hq, w.hkv, w.hd, w.F, w.eps)
    lw = _layer(w)
    xs = I.to_f64(I.residual_stream(w), "fp32")[0]
    a0, f0 = O.block(od, xs, O.Layer(lw), pos=np.arange(w.T))
    a1, f1 = O.block(od, xs, O.Layer(lw), pos=np.arange(w.T) + 37)
    np.testing.assert_allclose(a1, a0, rtol=0, atol=1e-11 * np.abs(a0).max())
    np.testing.assert_allclose(f1, f0, rtol=0, atol=1e-11 * np.abs(f0).max())


def test_qk_norm_unit_rms_and_scale_blindness():
    g = np.random.default_rng(4)
    heads, hd = 2, 32
    x = 5.0 * g.standard_normal((4, heads * hd))
    y = O.qk_transform(x, heads, hd, gain=np.ones(hd), eps=1e-12)
    np.testing.assert_allclose(np.sqrt((y.reshape(4, heads, hd) ** 2).mean(axis=2)), 1.0, rtol=1e-9)
    w = I.WORKLOADS["tiny_fp32"].replace(eps=1e-12)
    od = O.dims(w.B, w.T, w.d, w.hq, w.hkv, w.hd, w.F, w.eps)
    xs = I.to_f64(I.residual_stream(w), "fp32")[0]
    a0, _ = O.block(od, xs, O.Layer(_layer(w)))
    a1, _ = O.block(od, xs, O.Layer(_layer(w, wqk_scale=4.0)))   # exact in binary
    np.testing.assert_allclose(a1, a0, rtol=0, atol=1e-9 * np.abs(a0).max())


def test_sparse_layer_rotates_at_original_positions():
    w = I.WORKLOADS["tiny_fp32"].replace(B=1)
    od = O.dims(w.B, w.T, w.d, w.hq, w.hkv, w.hd, w.F, w.eps)
    lw = _layer(w)
    x = I.to_f64(I.residual_stream(w), "fp32")
    n = w.T // w.K
    # the same n token vectors, once at positions 0..n-1, once at 0, 2, 4, ...
    picked = x[0, :n].copy()
    xa = x.copy()
    xb = x.copy()
    xb[0, 0:2 * n:2] = picked
    bias_a = np.where(np.arange(w.T) < n, 50.0, -50.0)[None, :]
    bias_b = np.where((np.arange(w.T) < 2 * n) & (np.arange(w.T) % 2 == 0), 50.0, -50.0)[None, :]
    ya = O.layer_fwd(od, O.SPARSE, w.K, 0, O.Layer(lw), xa, bias=bias_a)
    yb = O.layer_fwd(od, O.SPARSE, w.K, 0, O.Layer(lw), xb, bias=bias_b)
    assert np.array_equal(yb["idx"][0], np.arange(0, 2 * n, 2))
    out_a = ya["y"][0, :n]
    out_b = yb["y"][0, 0:2 * n:2]
    assert np.abs(out_a - out_b).max() > 1e-6
    # and the layer is the block on the gathered rows at their original positions
    a, f = O.block(od, xb[0, 0:2 * n:2], O.Layer(lw), pos=np.arange(0, 2 * n, 2))
    r = 1.0 / (1.0 + np.exp(-yb["s"][0, 0:2 * n:2]))
    np.testing.assert_allclose(out_b, picked + float(lw["varsigma"]) * r[:, None] * (a + f),
                               rtol=0, atol=1e-12 * np.abs(out_b).max())
