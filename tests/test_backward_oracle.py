"""Pins of the oracle's layer backward (CPU only).

The backward is held against finite differences of the forward oracle (itself pinned
in test_oracle_pins.py): for J = sum(dy * y) + route_coef * L_route (Eq. 9 of the X-MoD
notes, section "top-k in training, causal threshold at evaluation"), the central
difference of J along a random direction of x, of every weight and of varsigma must
equal the inner product of that direction with the returned gradient. The selection is
held fixed on both sides (forced indices), as the backward holds it; with the optional
QK-norm gains and rotary embedding too. Plus closed forms: the skip path of unselected
rows, the Eq. 9 value at p = 1/2, an FFN with W_down = 0; for the Selected-Q / full-KV
control, the K = 1 case (every token selected: the sparse layer) and the rows that no
query sees.
"""
import numpy as np
import pytest

import oracle as O

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

B, T, d, HQ, HKV, HD, F, K = 2, 12, 16, 4, 2, 4, 24, 3
NAMES = ("w_r", "g1", "wq", "wk", "wv", "wo", "g2", "wg", "wu", "wd")


def _weights(g, scale=0.3):
    return {"w_r": g.standard_normal(d) / 4, "g1": 1 + 0.1 * g.standard_normal(d),
            "wq": g.standard_normal((HQ * HD, d)) * scale,
            "wk": g.standard_normal((HKV * HD, d)) * scale,
            "wv": g.standard_normal((HKV * HD, d)) * scale,
            "wo": g.standard_normal((d, HQ * HD)) * scale, "g2": 1 + 0.1 * g.standard_normal(d),
            "wg": g.standard_normal((F, d)) * scale, "wu": g.standard_normal((F, d)) * scale,
            "wd": g.standard_normal((d, F)) * scale}


def _objective(dm, kind, gate, W, vs, x, dy, bias, idx, coef):
    out = O.layer_fwd(dm, kind, K, gate, O.Layer(W, vs), x, bias=bias, idx_force=idx)
    val = float((dy * out["y"]).sum())
    if kind in (O.SPARSE, O.RFFN, O.FULLKV) and coef:
        s = out["s"]
        p = 1.0 / (1.0 + np.exp(-s))
        q = np.zeros_like(s)
        np.put_along_axis(q, idx, 1.0, 1)
        val += coef * float(-(q * np.log(p) + (1 - q) * np.log(1 - p)).mean())
    return val


@pytest.mark.parametrize("kind,gate,coef", [(O.SPARSE, O.GATE_XMOD, 0.0),
                                            (O.SPARSE, O.GATE_MOD, 0.0),
                                            (O.SPARSE, O.GATE_XMOD, 0.7),
                                            (O.SPARSE, O.GATE_MOD, 0.3),
                                            (O.DENSE, O.GATE_XMOD, 0.0)])
def test_layer_bwd_matches_finite_differences(kind, gate, coef):
    g = np.random.default_rng(10 + 3 * kind + gate)
    dm = O.dims(B, T, d, HQ, HKV, HD, F)
    W = _weights(g)
    vs = 0.8
    x = g.standard_normal((B, T, d))
    dy = g.standard_normal((B, T, d))
    bias = 0.1 * g.standard_normal((B, T))
    r = O.layer_bwd(dm, kind, K, gate, O.Layer(W, vs), x, dy, bias=bias, route_coef=coef)
    idx = r["idx"]
    eps = 1e-6

    def fd(x_=x, W_=W, vs_=vs):
        return _objective(dm, kind, gate, W_, vs_, x_, dy, bias, idx, coef)

    def check(num, ana, what):
        assert abs(num - ana) <= 1e-6 * max(1.0, abs(num)), f"{what}: fd {num} vs grad {ana}"

    v = g.standard_normal(x.shape)
    check((fd(x_=x + eps * v) - fd(x_=x - eps * v)) / (2 * eps), float((r["dx"] * v).sum()), "x")
    for name in NAMES:
        v = g.standard_normal(W[name].shape)
        Wp, Wm = dict(W), dict(W)
        Wp[name] = W[name] + eps * v
        Wm[name] = W[name] - eps * v
        check((fd(W_=Wp) - fd(W_=Wm)) / (2 * eps), float((r["grads"][name] * v).sum()), name)
    check((fd(vs_=vs + eps) - fd(vs_=vs - eps)) / (2 * eps), r["varsigma"], "varsigma")
    if kind == O.DENSE or gate == O.GATE_MOD:
        assert r["varsigma"] == 0.0
    if kind == O.DENSE:
        assert np.all(r["grads"]["w_r"] == 0.0)


def test_unselected_rows_pass_the_gradient_through():
    """With no Eq. 9 term, a token the layer skipped has y = x, so dx = dy exactly."""
    g = np.random.default_rng(3)
    dm = O.dims(B, T, d, HQ, HKV, HD, F)
    x = g.standard_normal((B, T, d))
    dy = g.standard_normal((B, T, d))
    r = O.layer_bwd(dm, O.SPARSE, K, O.GATE_XMOD, O.Layer(_weights(g), 1.1), x, dy)
    sel = np.zeros((B, T), bool)
    np.put_along_axis(sel, r["idx"], True, 1)
    np.testing.assert_array_equal(r["dx"][~sel], dy[~sel])
    assert np.any(r["dx"][sel] != dy[sel])


def test_route_loss_at_even_odds():
    """w_r = 0 and no bias give p = 1/2 for every token: L_route = ln 2, and the Eq. 9 term
    alone moves the logits by coef * (1/2 - q) / (B*T) each."""
    g = np.random.default_rng(4)
    dm = O.dims(B, T, d, HQ, HKV, HD, F)
    W = _weights(g)
    W["w_r"] = np.zeros(d)
    x = g.standard_normal((B, T, d))
    zero = np.zeros((B, T, d))
    coef = 5.0
    r = O.layer_bwd(dm, O.SPARSE, K, O.GATE_XMOD, O.Layer(W, 1.0), x, zero, route_coef=coef)
    assert r["route_loss"] == pytest.approx(np.log(2.0), rel=1e-14)
    q = np.zeros((B, T))
    np.put_along_axis(q, r["idx"], 1.0, 1)
    ds = coef * (0.5 - q) / (B * T)
    np.testing.assert_allclose(r["grads"]["w_r"], np.einsum("bt,btc->c", ds, x), rtol=1e-12)
    np.testing.assert_allclose(r["dx"], np.zeros_like(x), atol=0)   # w_r = 0: no path to x


def test_zero_down_projection():
    """W_down = 0 makes f = 0: no gradient reaches W_gate or W_up, while W_down's gradient
    is df^T H with H = silu(G) U, which is not zero."""
    g = np.random.default_rng(5)
    dm = O.dims(B, T, d, HQ, HKV, HD, F)
    W = _weights(g)
    W["wd"] = np.zeros((d, F))
    x = g.standard_normal((B, T, d))
    dy = g.standard_normal((B, T, d))
    r = O.layer_bwd(dm, O.SPARSE, K, O.GATE_MOD, O.Layer(W, 1.0), x, dy)
    assert np.all(r["grads"]["wg"] == 0.0) and np.all(r["grads"]["wu"] == 0.0)
    assert np.any(r["grads"]["wd"] != 0.0)


@pytest.mark.parametrize("kind,gq,gk,theta", [(O.SPARSE, True, True, 1e4), (O.SPARSE, False, True, 0.0),
                                              (O.SPARSE, True, False, 500.0),
                                              (O.DENSE, True, True, 1e4)])
def test_layer_bwd_qk_norm_rope_matches_finite_differences(kind, gq, gk, theta):
    """The Qwen3-style extras: QK-norm gains (their own gradients) and the rotary embedding
    at the tokens' original positions; central differences of the forward oracle along
    random directions of x, of the projections and of the gains."""
    g = np.random.default_rng(50 + 2 * kind + int(gq) + int(theta > 0))
    dm = O.dims(B, T, d, HQ, HKV, HD, F)
    W = _weights(g)
    if gq:
        W["gq"] = 1 + 0.2 * g.standard_normal(HD)
    if gk:
        W["gk"] = 1 + 0.2 * g.standard_normal(HD)
    W["rope_theta"] = theta
    vs = 1.1
    x = g.standard_normal((B, T, d))
    dy = g.standard_normal((B, T, d))
    bias = 0.1 * g.standard_normal((B, T))
    r = O.layer_bwd(dm, kind, K, O.GATE_XMOD, O.Layer(W, vs), x, dy, bias=bias, route_coef=0.2)
    idx = r["idx"]
    eps = 1e-6

    def J(x_=x, W_=W):
        return _objective(dm, kind, O.GATE_XMOD, W_, vs, x_, dy, bias, idx, 0.2)

    def check(num, ana, what):
        assert abs(num - ana) <= 1e-6 * max(1.0, abs(num)), f"{what}: fd {num} vs grad {ana}"

    v = g.standard_normal(x.shape)
    check((J(x_=x + eps * v) - J(x_=x - eps * v)) / (2 * eps), float((r["dx"] * v).sum()), "x")
    for name in ("wq", "wk", "wv", "g1", "w_r") + (("gq",) if gq else ()) + (("gk",) if gk else ()):
        if kind == O.DENSE and name == "w_r":
            continue
        v = g.standard_normal(np.shape(W[name]))
        Wp, Wm = dict(W), dict(W)
        Wp[name] = W[name] + eps * v
        Wm[name] = W[name] - eps * v
        check((J(W_=Wp) - J(W_=Wm)) / (2 * eps), float((r["grads"][name] * v).sum()), name)


@pytest.mark.parametrize("kind,gate,coef", [(O.ATTN, O.GATE_XMOD, 0.0), (O.RFFN, O.GATE_XMOD, 0.4),
                                            (O.RFFN, O.GATE_MOD, 0.0)])
def test_variant_layer_bwd_matches_finite_differences(kind, gate, coef):
    """The mechanism controls' halves: FullAttn (attention on every token, y = x + a) and
    Routed-FFN (the FFN half on the top-(T/K) tokens with a = 0 in the gated residual)."""
    g = np.random.default_rng(70 + kind + gate)
    dm = O.dims(B, T, d, HQ, HKV, HD, F)
    W = _weights(g)
    vs = 0.9
    x = g.standard_normal((B, T, d))
    dy = g.standard_normal((B, T, d))
    bias = 0.1 * g.standard_normal((B, T))
    r = O.layer_bwd(dm, kind, K, gate, O.Layer(W, vs), x, dy, bias=bias, route_coef=coef)
    idx = r["idx"]
    eps = 1e-6

    def J(x_=x, W_=W, vs_=vs):
        return _objective(dm, kind, gate, W_, vs_, x_, dy, bias, idx, coef)

    def check(num, ana, what):
        assert abs(num - ana) <= 1e-6 * max(1.0, abs(num)), f"{what}: fd {num} vs grad {ana}"

    v = g.standard_normal(x.shape)
    check((J(x_=x + eps * v) - J(x_=x - eps * v)) / (2 * eps), float((r["dx"] * v).sum()), "x")
    for name in NAMES:
        v = g.standard_normal(W[name].shape)
        Wp, Wm = dict(W), dict(W)
        Wp[name] = W[name] + eps * v
        Wm[name] = W[name] - eps * v
        check((J(W_=Wp) - J(W_=Wm)) / (2 * eps), float((r["grads"][name] * v).sum()), name)
    check((J(vs_=vs + eps) - J(vs_=vs - eps)) / (2 * eps), r["varsigma"], "varsigma")
    unused = ("g2", "wg", "wu", "wd", "w_r") if kind == O.ATTN else ("g1", "wq", "wk", "wv", "wo")
    for name in unused:
        assert np.all(r["grads"][name] == 0.0), name



@pytest.mark.parametrize("gate,coef,extras", [(O.GATE_XMOD, 0.0, False), (O.GATE_MOD, 0.5, False),
                                              (O.GATE_XMOD, 0.3, True)])
def test_fullkv_layer_bwd_matches_finite_differences(gate, coef, extras):
    """Selected-Q / full-KV control (X-MoD notes, "mechanism controls"): the selected tokens
    are the queries, every token provides keys and values, so the gradient reaches the
    unselected rows through k and v; central differences of the forward oracle along random
    directions of x, of every weight and of varsigma, the selection held fixed."""
    g = np.random.default_rng(90 + gate + 2 * int(extras))
    dm = O.dims(B, T, d, HQ, HKV, HD, F)
    W = _weights(g)
    if extras:
        W["gq"] = 1 + 0.2 * g.standard_normal(HD)
        W["gk"] = 1 + 0.2 * g.standard_normal(HD)
        W["rope_theta"] = 1e4
    vs = 0.9
    x = g.standard_normal((B, T, d))
    dy = g.standard_normal((B, T, d))
    bias = 0.1 * g.standard_normal((B, T))
    r = O.layer_bwd(dm, O.FULLKV, K, gate, O.Layer(W, vs), x, dy, bias=bias, route_coef=coef)
    idx = r["idx"]
    eps = 1e-6

    def J(x_=x, W_=W, vs_=vs):
        return _objective(dm, O.FULLKV, gate, W_, vs_, x_, dy, bias, idx, coef)

    def check(num, ana, what):
        assert abs(num - ana) <= 1e-6 * max(1.0, abs(num)), f"{what}: fd {num} vs grad {ana}"

    v = g.standard_normal(x.shape)
    check((J(x_=x + eps * v) - J(x_=x - eps * v)) / (2 * eps), float((r["dx"] * v).sum()), "x")
    names = NAMES + (("gq", "gk") if extras else ())
    for name in names:
        v = g.standard_normal(np.shape(W[name]))
        Wp, Wm = dict(W), dict(W)
        Wp[name] = W[name] + eps * v
        Wm[name] = W[name] - eps * v
        check((J(W_=Wp) - J(W_=Wm)) / (2 * eps), float((r["grads"][name] * v).sum()), name)
    check((J(vs_=vs + eps) - J(vs_=vs - eps)) / (2 * eps), r["varsigma"], "varsigma")


@pytest.mark.parametrize("gate", [O.GATE_XMOD, O.GATE_MOD])
def test_fullkv_with_every_token_selected_is_the_sparse_layer(gate):
    """K = 1 selects every token: the queries are all rows and the keys are the same rows,
    so the full-KV layer and the sparse layer are one function, gradients included."""
    g = np.random.default_rng(95 + gate)
    dm = O.dims(B, T, d, HQ, HKV, HD, F)
    W = _weights(g)
    W["gk"] = 1 + 0.2 * g.standard_normal(HD)
    W["rope_theta"] = 500.0
    x = g.standard_normal((B, T, d))
    dy = g.standard_normal((B, T, d))
    bias = 0.1 * g.standard_normal((B, T))
    a = O.layer_bwd(dm, O.FULLKV, 1, gate, O.Layer(W, 1.2), x, dy, bias=bias, route_coef=0.4)
    b = O.layer_bwd(dm, O.SPARSE, 1, gate, O.Layer(W, 1.2), x, dy, bias=bias, route_coef=0.4)
    np.testing.assert_allclose(a["dx"], b["dx"], rtol=1e-11, atol=1e-12)
    for name in a["grads"]:
        np.testing.assert_allclose(a["grads"][name], b["grads"][name], rtol=1e-11, atol=1e-12,
                                   err_msg=name)
    assert a["varsigma"] == pytest.approx(b["varsigma"], rel=1e-11)
    assert a["route_loss"] == pytest.approx(b["route_loss"], rel=1e-14)


def test_fullkv_rows_no_query_sees():
    """Without Eq. 9, a token after the sequence's last selected position is no query's key
    and is not selected: its dx is dy exactly. With W_k = W_v = 0 no gradient reaches any
    unselected row (the keys and values are zero whatever the row holds); with the weights
    nonzero, unselected rows before the last selected position do receive one."""
    g = np.random.default_rng(97)
    dm = O.dims(B, T, d, HQ, HKV, HD, F)
    W = _weights(g)
    x = g.standard_normal((B, T, d))
    dy = g.standard_normal((B, T, d))
    r = O.layer_bwd(dm, O.FULLKV, K, O.GATE_XMOD, O.Layer(W, 1.1), x, dy)
    sel = np.zeros((B, T), bool)
    np.put_along_axis(sel, r["idx"], True, 1)
    after = np.arange(T)[None, :] > r["idx"].max(axis=1, keepdims=True)
    before = ~sel & ~after
    assert after.any()
    np.testing.assert_array_equal(r["dx"][after], dy[after])
    assert before.any() and np.all(np.any(r["dx"][before] != dy[before], axis=-1))
    W["wk"] = np.zeros_like(W["wk"])
    W["wv"] = np.zeros_like(W["wv"])
    r0 = O.layer_bwd(dm, O.FULLKV, K, O.GATE_XMOD, O.Layer(W, 1.1), x, dy)
    np.testing.assert_array_equal(r0["dx"][~sel], dy[~sel])
