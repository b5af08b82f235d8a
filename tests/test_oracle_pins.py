"""Pins of the CPU oracle's numerics against closed forms, special cases and brute force.

The pages print no worked numeric example of a layer, so each step of the oracle
is pinned by a property that a plausible mistake (dropped term, wrong sign,
transposed operand, off-by-one mask, wrong head map, wrong gate placement)
would break.
"""
import itertools
import math

import numpy as np
import pytest

import oracle as O
from sparse_depth_token_gb300 import inputs as I


def _rng(seed=0):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- router (Eq. 8)

def test_router_one_hot_and_bias():
    d = 16
    w = _rng().standard_normal(d)
    x = np.eye(d)
    b = np.linspace(-1, 1, d)
    s, r = O.router(x, w, b)
    np.testing.assert_array_equal(s, w + b)


def test_router_sigmoid_closed_forms():
    d = 4
    w = np.array([1.0, 0, 0, 0])
    x = np.array([[0.0, 5, 5, 5], [math.log(3), 0, 0, 0], [-math.log(3), 0, 0, 0], [40.0, 0, 0, 0]])
    s, r = O.router(x, w)
    assert r[0] == 0.5                       # sigmoid(0)
    assert abs(r[1] - 0.75) < 1e-15          # sigmoid(ln 3) = 3/4
    assert abs(r[2] - 0.25) < 1e-15          # sigmoid(-ln 3) = 1/4
    assert r[3] == 1.0                       # saturates exactly in double


def test_router_linear_in_x_without_bias():
    d = 32
    g = _rng(1)
    w, x = g.standard_normal(d), g.standard_normal((5, d))
    s1, _ = O.router(x, w)
    s2, _ = O.router(2.0 * x, w)
    np.testing.assert_allclose(s2, 2 * s1, rtol=1e-14, atol=1e-14)
    s3, _ = O.router(x, -w)
    np.testing.assert_allclose(s3, -s1, rtol=1e-14, atol=1e-14)


# ---------------------------------------------------------------- top-(T/K)

def _brute_topk(s, k):
    """Enumerate every k-subset; keep the one whose sorted logits are largest, ties going
    to the subset with the smaller positions (lexicographic on ascending positions)."""
    T = len(s)
    best = None
    for sub in itertools.combinations(range(T), k):
        key = (sorted((s[i] for i in sub), reverse=True), [-i for i in sub])
        if best is None or key > best[0]:
            best = (key, sub)
    return list(best[1])


@pytest.mark.parametrize("T,K", [(8, 2), (9, 3), (10, 4), (6, 1), (7, 7), (10, 3)])
def test_topk_brute_force_random(T, K):
    g = _rng(T * 10 + K)
    for trial in range(20):
        s = g.standard_normal(T)
        if trial % 3 == 1:  # duplicated values around the k-th rank
            s = np.round(s * 2) / 2
        if trial % 3 == 2:
            s = g.integers(-1, 2, T).astype(float)
        k = T // K
        assert O.topk(s[None, :], k)[0].tolist() == _brute_topk(list(s), k)


def test_topk_ties_lower_position_and_signed_zero():
    assert O.topk(np.zeros((1, 8)), 3)[0].tolist() == [0, 1, 2]
    s = np.array([[-0.0, 0.0, -0.0, 0.0, -1.0, 1.0]])
    assert O.topk(s, 3)[0].tolist() == [0, 1, 5]     # -0 == +0: positions decide
    s = np.array([[1.0, 2.0, 2.0, 0.5, 2.0, 2.0]])
    assert O.topk(s, 3)[0].tolist() == [1, 2, 4]


def test_topk_exact_count_and_order():
    g = _rng(3)
    B, T = 3, 64
    s = g.standard_normal((B, T))
    for K in (1, 2, 3, 4, 8, 16, 64):
        n = T // K
        idx = O.topk(s, n)
        assert idx.shape == (B, n)
        for b in range(B):
            assert np.all(np.diff(idx[b]) > 0)
            chosen = set(idx[b].tolist())
            kth = min(s[b, list(chosen)])
            assert all(s[b, t] <= kth for t in range(T) if t not in chosen)


def test_topk_rejects_nonfinite():
    with pytest.raises(ValueError):
        O.topk(np.array([[0.0, np.nan, 1.0]]), 1)
    with pytest.raises(ValueError):
        O.topk(np.array([[0.0, np.inf, 1.0]]), 1)


# ---------------------------------------------------------------- RMSNorm, linear

def test_rmsnorm_closed_forms():
    d = 64
    for c in (3.0, -0.25):
        out = O.rmsnorm(np.full((1, d), c), np.ones(d), 0.0)
        np.testing.assert_allclose(out, np.sign(c), rtol=1e-15)
        eps = 1e-2
        out = O.rmsnorm(np.full((1, d), c), np.ones(d), eps)
        np.testing.assert_allclose(out, c / math.sqrt(c * c + eps), rtol=1e-14)
    x = np.zeros((1, d))
    x[0, 5] = math.sqrt(d)                    # mean square 1
    gamma = np.arange(d, dtype=float)
    out = O.rmsnorm(x, gamma, 0.0)
    assert out[0, 5] == pytest.approx(math.sqrt(d) * 5, rel=1e-15)
    assert np.count_nonzero(out) == 1


def test_rmsnorm_scale_invariant():
    g = _rng(4)
    x = g.standard_normal((3, 40))
    gam = g.standard_normal(40)
    np.testing.assert_allclose(O.rmsnorm(7.5 * x, gam, 0.0), O.rmsnorm(x, gam, 0.0), rtol=1e-13)


def test_linear_orientation():
    g = _rng(5)
    x = g.standard_normal((4, 6))
    W = np.zeros((3, 6))          # [out=3, in=6]
    W[2, 4] = 1.0
    W[0, 1] = -2.0
    y = O.linear(x, W)
    assert y.shape == (4, 3)
    np.testing.assert_array_equal(y[:, 2], x[:, 4])
    np.testing.assert_array_equal(y[:, 0], -2.0 * x[:, 1])
    np.testing.assert_array_equal(y[:, 1], 0.0)
    np.testing.assert_array_equal(O.linear(x, np.eye(6)), x)


# ---------------------------------------------------------------- causal GQA attention

def test_attention_single_token_and_first_row():
    g = _rng(6)
    hq, hkv, hd = 4, 2, 8
    for n in (1, 5):
        q = g.standard_normal((n, hq * hd))
        k = g.standard_normal((n, hkv * hd))
        v = g.standard_normal((n, hkv * hd))
        o = O.attention(q, k, v, hq, hkv, hd)
        for h in range(hq):
            kv = h // (hq // hkv)
            np.testing.assert_allclose(o[0, h * hd:(h + 1) * hd], v[0, kv * hd:(kv + 1) * hd],
                                       rtol=1e-15)


def test_attention_zero_query_is_causal_running_mean():
    g = _rng(7)
    n, hq, hkv, hd = 9, 6, 3, 4
    q = np.zeros((n, hq * hd))
    k = g.standard_normal((n, hkv * hd))
    v = g.standard_normal((n, hkv * hd))
    o = O.attention(q, k, v, hq, hkv, hd)
    G = hq // hkv
    for i in range(n):
        for h in range(hq):
            kv = h // G
            np.testing.assert_allclose(o[i, h * hd:(h + 1) * hd],
                                       v[:i + 1, kv * hd:(kv + 1) * hd].mean(axis=0), rtol=1e-13)


def test_attention_gqa_head_map():
    n, hq, hkv, hd = 3, 8, 2, 4
    g = _rng(8)
    q = g.standard_normal((n, hq * hd))
    k = g.standard_normal((n, hkv * hd))
    v = np.zeros((n, hkv * hd))
    v[:, :hd] = 10.0        # KV head 0
    v[:, hd:] = -3.0        # KV head 1
    o = O.attention(q, k, v, hq, hkv, hd)
    for h in range(hq):
        expect = 10.0 if h < hq // hkv else -3.0
        np.testing.assert_allclose(o[:, h * hd:(h + 1) * hd], expect, rtol=1e-14)


def test_attention_two_key_closed_form():
    """Row 1 weights key 1 by sigmoid((q.k1 - q.k0)/sqrt(hd)): pins the scale and exp base."""
    hd = 16
    g = _rng(9)
    q = g.standard_normal((2, hd))
    k = g.standard_normal((2, hd))
    v = g.standard_normal((2, hd))
    o = O.attention(q, k, v, 1, 1, hd)
    delta = (q[1] @ k[1] - q[1] @ k[0]) / math.sqrt(hd)
    w1 = 1.0 / (1.0 + math.exp(-delta))
    np.testing.assert_allclose(o[1], v[0] + w1 * (v[1] - v[0]), rtol=1e-12, atol=1e-14)


def test_attention_future_keys_masked():
    g = _rng(10)
    n, hd = 6, 8
    q = g.standard_normal((n, hd))
    k = g.standard_normal((n, hd))
    v = g.standard_normal((n, hd))
    o1 = O.attention(q, k, v, 1, 1, hd)
    k2, v2 = k.copy(), v.copy()
    k2[4:] *= 100.0
    v2[4:] = 1e6
    o2 = O.attention(q, k2, v2, 1, 1, hd)
    np.testing.assert_array_equal(o1[:4], o2[:4])
    assert np.all(np.abs(o2[4:]) > 1e3)


def test_attention_row_subset_matches_full():
    g = _rng(11)
    n, hq, hkv, hd = 12, 4, 1, 8
    q, k, v = (g.standard_normal((n, h * hd)) for h in (hq, hkv, hkv))
    full = O.attention(q, k, v, hq, hkv, hd)
    rows = [11, 0, 7]
    sub = O.attention(q, k, v, hq, hkv, hd, rows=rows)
    np.testing.assert_array_equal(sub, full[rows])


# ---------------------------------------------------------------- block, layer, residual gates

def _layer_arrays(g, d, hq, hkv, hd, F, std=0.1):
    return {"w_r": g.standard_normal(d) / math.sqrt(d), "g1": np.ones(d), "g2": np.ones(d),
            "wq": g.standard_normal((hq * hd, d)) * std, "wk": g.standard_normal((hkv * hd, d)) * std,
            "wv": g.standard_normal((hkv * hd, d)) * std, "wo": g.standard_normal((d, hq * hd)) * std,
            "wg": g.standard_normal((F, d)) * std, "wu": g.standard_normal((F, d)) * std,
            "wd": g.standard_normal((d, F)) * std}


def test_block_ffn_closed_form_scalar_path():
    """d_ff = 1, Wv = 0 (so a = 0): f = Wd * silu(Wg.v2) * (Wu.v2) with v2 = RMSNorm(x)."""
    d, hq, hkv, hd, F = 8, 2, 1, 4, 1
    g = _rng(12)
    arr = _layer_arrays(g, d, hq, hkv, hd, F)
    arr["wv"][:] = 0.0
    c = 2.0
    xs = np.full((3, d), c)                  # RMSNorm(const) = 1 per element (eps tiny)
    arr["wg"][:] = 0.125                     # Wg.v2 = 8 * 0.125 = 1
    arr["wu"][:] = -0.25                     # Wu.v2 = -2
    arr["wd"][:, 0] = np.arange(d)
    dm = O.dims(1, 3, d, hq, hkv, hd, F, eps=0.0)
    a, f = O.block(dm, xs, O.Layer(arr))
    np.testing.assert_array_equal(a, 0.0)
    silu1 = 1.0 / (1.0 + math.exp(-1.0))
    np.testing.assert_allclose(f, np.tile(np.arange(d) * silu1 * -2.0, (3, 1)), rtol=1e-14)


def test_block_zero_up_gives_zero_ffn_and_zero_wo_gives_zero_attn():
    d, hq, hkv, hd, F = 16, 4, 2, 4, 24
    g = _rng(13)
    arr = _layer_arrays(g, d, hq, hkv, hd, F)
    xs = g.standard_normal((7, d))
    dm = O.dims(1, 7, d, hq, hkv, hd, F)
    arr0 = dict(arr, wu=np.zeros_like(arr["wu"]))
    a, f = O.block(dm, xs, O.Layer(arr0))
    np.testing.assert_array_equal(f, 0.0)
    assert np.abs(a).max() > 1e-3
    arr1 = dict(arr, wo=np.zeros_like(arr["wo"]))
    a1, f1 = O.block(dm, xs, O.Layer(arr1))
    np.testing.assert_array_equal(a1, 0.0)
    # with a = 0 the FFN sees RMSNorm(xs) itself: compare to a block whose attention is zero
    arr2 = dict(arr, wv=np.zeros_like(arr["wv"]))
    a2, f2 = O.block(dm, xs, O.Layer(arr2))
    np.testing.assert_array_equal(a2, 0.0)
    np.testing.assert_array_equal(f1, f2)


def test_block_ffn_reads_the_in_block_residual_x_plus_a():
    """The FFN's input is RMSNorm(h)·γ2 with h = x_sel + a, a the attention residual
    (X-MoD notes, Eq. 6 / Eq. 7: a and f are the block's two residual branches; pre-norm
    SwiGLU block). Built so that every value is fixed by hand:
      rows x_i = 4·e_i, eps = 0        -> u_i = RMSNorm(x_i) = 2√2·e_i, Σ_j u_i[j] = 2√2;
      every Wv row constant c_j / (2√2) -> v = c = e_0 on every row, so each head's
                                          softmax average is c whatever the weights;
      Wo[:, 0] = Wo[:, hd] = 1          -> a = 2 on every element;
      h_i = x_i + a = 6 at i, 2 elsewhere -> mean(h²) = 8, v2 = h / (2√2);
      Wg = 1/√2 everywhere              -> Wg·v2 = (6 + 7·2) / 4 = 5 (row independent);
      Wu = √2 on column 0 only          -> Wu·v2 = 3 on row 0, 1 on rows 1, 2;
      f_i = Wd[:, 0]·silu(5)·(Wu·v2).
    An FFN fed RMSNorm(x_sel) gives Wg·v2 = 2, one fed RMSNorm(a) gives 4√2."""
    d, hq, hkv, hd, F, n = 8, 2, 1, 4, 1, 3
    g = _rng(21)
    s2 = math.sqrt(2.0)
    arr = {"w_r": np.zeros(d), "g1": np.ones(d), "g2": np.ones(d),
           "wq": g.standard_normal((hq * hd, d)), "wk": g.standard_normal((hkv * hd, d))}
    c = np.array([1.0, 0.0, 0.0, 0.0])
    arr["wv"] = np.repeat(c[:, None] / (2 * s2), d, axis=1)
    wo = np.zeros((d, hq * hd))
    wo[:, 0] = 1.0
    wo[:, hd] = 1.0
    arr["wo"] = wo
    arr["wg"] = np.full((F, d), 1.0 / s2)
    wu = np.zeros((F, d))
    wu[0, 0] = s2
    arr["wu"] = wu
    arr["wd"] = np.arange(1.0, d + 1)[:, None]
    xs = 4.0 * np.eye(d)[:n]
    dm = O.dims(1, n, d, hq, hkv, hd, F, eps=0.0)
    a, f = O.block(dm, xs, O.Layer(arr))
    np.testing.assert_allclose(a, 2.0, rtol=1e-14)
    silu5 = 5.0 / (1.0 + math.exp(-5.0))
    up = np.array([3.0, 1.0, 1.0])
    want = up[:, None] * silu5 * np.arange(1.0, d + 1)[None, :]
    np.testing.assert_allclose(f, want, rtol=1e-13)


def test_block_row_subset_matches_full():
    d, hq, hkv, hd, F = 16, 4, 2, 4, 24
    g = _rng(14)
    arr = _layer_arrays(g, d, hq, hkv, hd, F)
    xs = g.standard_normal((10, d))
    dm = O.dims(1, 10, d, hq, hkv, hd, F)
    L = O.Layer(arr)
    a, f = O.block(dm, xs, L)
    rows = [9, 2, 5]
    a2, f2 = O.block(dm, xs, L, rows=rows)
    np.testing.assert_array_equal(a2, a[rows])
    np.testing.assert_array_equal(f2, f[rows])


def _small_dims(B=2, T=16, d=16, hq=4, hkv=2, hd=4, F=24):
    return O.dims(B, T, d, hq, hkv, hd, F)


def test_sparse_layer_skip_identity_and_count():
    dm = _small_dims()
    g = _rng(15)
    L = O.Layer(_layer_arrays(g, dm.d, dm.hq, dm.hkv, dm.hd, dm.F), varsigma=0.7)
    x = g.standard_normal((dm.B, dm.T, dm.d))
    for K in (2, 3, 4):
        out = O.layer_fwd(dm, O.SPARSE, K, O.GATE_XMOD, L, x)
        n = dm.T // K
        changed = np.any(out["y"] != x, axis=-1)
        for b in range(dm.B):
            sel = out["idx"][b]
            assert len(sel) == n and np.all(np.diff(sel) > 0)
            assert set(np.nonzero(changed[b])[0].tolist()) <= set(sel.tolist())
            unsel = [t for t in range(dm.T) if t not in set(sel.tolist())]
            np.testing.assert_array_equal(out["y"][b, unsel], x[b, unsel])   # bitwise skip path
        np.testing.assert_array_equal(out["r_sel"], np.take_along_axis(out["r"], out["idx"], 1))


def test_eq6_eq7_gate_placement():
    """With f = 0 (W_up = 0): Eq. 6 gives x + a, Eq. 7 gives x + varsigma*r*a."""
    dm = _small_dims()
    g = _rng(16)
    arr = _layer_arrays(g, dm.d, dm.hq, dm.hkv, dm.hd, dm.F)
    arr["wu"][:] = 0.0
    vs = 1.3
    L = O.Layer(arr, varsigma=vs)
    x = g.standard_normal((dm.B, dm.T, dm.d))
    K = 4
    y6 = O.layer_fwd(dm, O.SPARSE, K, O.GATE_MOD, L, x)
    y7 = O.layer_fwd(dm, O.SPARSE, K, O.GATE_XMOD, L, x)
    np.testing.assert_array_equal(y6["idx"], y7["idx"])
    for b in range(dm.B):
        for j, t in enumerate(y6["idx"][b]):
            a = y6["y"][b, t] - x[b, t]
            np.testing.assert_allclose(y7["y"][b, t] - x[b, t], vs * y6["r_sel"][b, j] * a,
                                       rtol=1e-12, atol=1e-15)
    # and with the FFN live, Eq. 6 gates only f: x + a + r f
    arr2 = _layer_arrays(_rng(17), dm.d, dm.hq, dm.hkv, dm.hd, dm.F)
    L2 = O.Layer(arr2, varsigma=vs)
    arr2_nof = dict(arr2, wu=np.zeros_like(arr2["wu"]))
    L2_nof = O.Layer(arr2_nof, varsigma=vs)
    y_full = O.layer_fwd(dm, O.SPARSE, K, O.GATE_MOD, L2, x)
    y_a = O.layer_fwd(dm, O.SPARSE, K, O.GATE_MOD, L2_nof, x)
    y_x = O.layer_fwd(dm, O.SPARSE, K, O.GATE_XMOD, L2, x)
    for b in range(dm.B):
        for j, t in enumerate(y_full["idx"][b]):
            a = y_a["y"][b, t] - x[b, t]
            r = y_full["r_sel"][b, j]
            f = (y_full["y"][b, t] - x[b, t] - a) / r
            np.testing.assert_allclose(y_x["y"][b, t], x[b, t] + vs * r * (a + f), rtol=1e-10,
                                       atol=1e-12)


def test_sparse_k1_saturated_gate_equals_dense():
    """K = 1 selects every token; a bias of 40 makes r == 1.0 exactly in double; with
    varsigma = 1 Eq. 7 is then the dense update x + a + f."""
    dm = _small_dims()
    g = _rng(18)
    L = O.Layer(_layer_arrays(g, dm.d, dm.hq, dm.hkv, dm.hd, dm.F), varsigma=1.0)
    x = g.standard_normal((dm.B, dm.T, dm.d))
    bias = np.full((dm.B, dm.T), 40.0)
    ys = O.layer_fwd(dm, O.SPARSE, 1, O.GATE_XMOD, L, x, bias=bias)
    assert np.all(ys["r"] == 1.0)
    yd = O.layer_fwd(dm, O.DENSE, 1, O.GATE_XMOD, L, x)
    np.testing.assert_allclose(ys["y"], yd["y"], rtol=0, atol=1e-14)


def test_sparse_attention_only_among_selected():
    """Changing an unselected token (but keeping it unselected) leaves every output row unchanged."""
    dm = _small_dims(B=1, T=16)
    g = _rng(19)
    arr = _layer_arrays(g, dm.d, dm.hq, dm.hkv, dm.hd, dm.F)
    L = O.Layer(arr)
    x = g.standard_normal((1, dm.T, dm.d))
    out = O.layer_fwd(dm, O.SPARSE, 4, O.GATE_XMOD, L, x)
    unsel = [t for t in range(dm.T) if t not in set(out["idx"][0].tolist())]
    x2 = x.copy()
    x2[0, unsel[0]] *= 0.5     # smaller norm never raises |s| above the k-th for this row...
    out2 = O.layer_fwd(dm, O.SPARSE, 4, O.GATE_XMOD, L, x2, idx_force=out["idx"])
    sel = out["idx"][0]
    np.testing.assert_array_equal(out2["y"][0, sel], out["y"][0, sel])


def test_layer_row_mask_matches_full():
    dm = _small_dims(B=2, T=20)
    g = _rng(20)
    L = O.Layer(_layer_arrays(g, dm.d, dm.hq, dm.hkv, dm.hd, dm.F), varsigma=0.9)
    x = g.standard_normal((dm.B, dm.T, dm.d))
    mask = np.zeros((dm.B, dm.T), dtype=np.int32)
    mask[0, [3, 19]] = 1
    mask[1, 7] = 1
    for kind in (O.SPARSE, O.DENSE):
        full = O.layer_fwd(dm, kind, 4, O.GATE_XMOD, L, x)
        part = O.layer_fwd(dm, kind, 4, O.GATE_XMOD, L, x, row_mask=mask)
        m = mask.astype(bool)
        np.testing.assert_array_equal(part["y"][m], full["y"][m])


def test_stack_equals_layer_sequence_and_seq_mask():
    from oracle import structure as S
    dm = _small_dims(B=2, T=16)
    g = _rng(21)
    kinds = S.schedule(1, 1, 1, 4)
    Ls = [O.Layer(_layer_arrays(g, dm.d, dm.hq, dm.hkv, dm.hd, dm.F), varsigma=0.8) for _ in kinds]
    x = g.standard_normal((dm.B, dm.T, dm.d))
    bias = g.standard_normal((dm.B, dm.T)) * 0.1
    y = O.stack_fwd(dm, 4, O.GATE_XMOD, kinds, Ls, x, bias=bias)
    z = x.copy()
    for k, L in zip(kinds, Ls):
        z = O.layer_fwd(dm, k, 4, O.GATE_XMOD, L, z, bias=bias)["y"]
    np.testing.assert_array_equal(y, z)
    ym = O.stack_fwd(dm, 4, O.GATE_XMOD, kinds, Ls, x, bias=bias, seq_mask=np.array([0, 1]))
    np.testing.assert_array_equal(ym[1], y[1])
    np.testing.assert_array_equal(ym[0], x[0])


# ---------------------------------------------------------------- bf16 mirroring

def test_round_bf16_ties_to_even():
    assert O.round_bf16(1.0 + 2.0 ** -8) == 1.0
    assert O.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert O.round_bf16(-(1.0 + 3 * 2.0 ** -8)) == -(1.0 + 2.0 ** -6)
    assert O.round_bf16(1.0 + 2.0 ** -8 + 2.0 ** -30) == 1.0 + 2.0 ** -7
    assert O.round_bf16(0.0) == 0.0


def test_round_bf16_agrees_with_float32_path():
    """Independent implementation check: for float32-representable values the oracle's
    rounding equals the generator's float32 -> bf16 conversion."""
    g = _rng(22)
    v = (g.standard_normal(2000) * 10.0 ** g.integers(-3, 4, 2000)).astype(np.float32)
    ref = I.bf16_bits_to_f32(I.f32_to_bf16_bits(v)).astype(np.float64)
    got = np.array([O.round_bf16(float(t)) for t in v])
    np.testing.assert_array_equal(got, ref)


def test_round_bf16_array_matches_scalar_and_stack_mirroring():
    g = _rng(23)
    v = g.standard_normal((3, 5, 7)) * 10.0 ** g.integers(-3, 4, (3, 5, 7))
    got = O.round_bf16_array(v)
    assert got.shape == v.shape
    np.testing.assert_array_equal(got.ravel(), [O.round_bf16(float(t)) for t in v.ravel()])
    # one dense layer in storage-mirroring mode = the layer, then the rounding
    d, hq, hkv, hd, F = 16, 4, 2, 4, 24
    arr = _layer_arrays(_rng(24), d, hq, hkv, hd, F)
    x = g.standard_normal((2, 6, d))
    dm = O.dims(2, 6, d, hq, hkv, hd, F)
    y = O.layer_fwd(dm, O.DENSE, 1, 0, O.Layer(arr), x)["y"]
    mirrored = O.stack_fwd(dm, 1, 0, [O.DENSE], [O.Layer(arr)], x, mirror_bf16=True)
    np.testing.assert_array_equal(O.round_bf16_array(y), mirrored)


def test_gated_scatter_matches_layer_residual():
    """The standalone scatter step reproduces the layer's own residual on its selected rows."""
    dm = _small_dims()
    g = _rng(23)
    L = O.Layer(_layer_arrays(g, dm.d, dm.hq, dm.hkv, dm.hd, dm.F), varsigma=1.1)
    x = g.standard_normal((dm.B, dm.T, dm.d))
    K = 4
    for gate in (O.GATE_XMOD, O.GATE_MOD):
        out = O.layer_fwd(dm, O.SPARSE, K, gate, L, x)
        n = dm.T // K
        rows = (np.arange(dm.B)[:, None] * dm.T + out["idx"]).reshape(-1)
        a, f = [], []
        for b in range(dm.B):
            ab, fb = O.block(dm, x[b, out["idx"][b]], L)
            a.append(ab)
            f.append(fb)
        a, f = np.concatenate(a), np.concatenate(f)
        y = O.gated_scatter(x.reshape(-1, dm.d), rows, a, f, out["r_sel"].reshape(-1), 1.1, gate)
        np.testing.assert_array_equal(y.reshape(x.shape), out["y"])
        if gate == O.GATE_XMOD:   # a + f passed pre-summed
            y2 = O.gated_scatter(x.reshape(-1, dm.d), rows, a + f, None, out["r_sel"].reshape(-1),
                                 1.1, gate)
            np.testing.assert_allclose(y2.reshape(x.shape), out["y"], rtol=1e-14, atol=1e-14)
