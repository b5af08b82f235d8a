"""The oracle's Routed-FFN halves (X-MoD notes, "mechanism controls": full-sequence
attention modules, and FFN-only refinements of the top-(T/K) tokens) pinned to the
dense layer through cases where the missing half is exactly zero:
  * a FullAttn layer equals the dense layer whose up projection is zero (f = 0);
  * a routed FFN layer with K = 1, an overwhelming bias (every gate exactly 1) and
    varsigma = 1 equals the dense layer whose output projection is zero (a = 0);
  * a routed FFN layer selects what the sparse layer with the same router selects."""
import numpy as np

import oracle as O
from sparse_depth_token_gb300 import inputs as I


def _setup(**over):
    w = I.WORKLOADS["tiny_fp32"].replace(**over)
    lw = I.layer_weights(w, 2)
    od = O.dims(w.B, w.T, w.d, w.hq, w.hkv, w.hd, w.F, w.eps)
    x = I.to_f64(I.residual_stream(w), "fp32")
    return w, lw, od, x


def test_full_attention_layer_is_dense_without_ffn():
    w, lw, od, x = _setup()
    y = O.layer_fwd(od, O.ATTN, w.K, 0, O.Layer(lw), x)["y"]
    ref = O.layer_fwd(od, O.DENSE, w.K, 0, O.Layer(dict(lw, wu=np.zeros_like(lw["wu"]))), x)["y"]
    assert np.array_equal(y, ref)
    assert not np.array_equal(y, x)


def test_routed_ffn_with_unit_gates_is_dense_without_attention():
    w, lw, od, x = _setup()
    lw = dict(lw, varsigma=np.float32(1.0))
    bias = np.full((w.B, w.T), 1e3)
    y = O.layer_fwd(od, O.RFFN, 1, 0, O.Layer(lw), x, bias=bias)["y"]
    ref = O.layer_fwd(od, O.DENSE, 1, 0, O.Layer(dict(lw, wo=np.zeros_like(lw["wo"]))), x)["y"]
    assert np.array_equal(y, ref)


def test_routed_ffn_selects_like_the_sparse_layer():
    w, lw, od, x = _setup()
    bias = I.router_bias(w)
    a = O.layer_fwd(od, O.RFFN, w.K, 0, O.Layer(lw), x, bias=bias)
    b = O.layer_fwd(od, O.SPARSE, w.K, 0, O.Layer(lw), x, bias=bias)
    assert np.array_equal(a["idx"], b["idx"])
    assert np.allclose(a["r_sel"], b["r_sel"], rtol=0, atol=0)
    sel = np.zeros((w.B, w.T), bool)
    np.put_along_axis(sel, a["idx"], True, 1)
    x3 = x.reshape(w.B, w.T, w.d)
    assert np.array_equal(a["y"].reshape(x3.shape)[~sel], x3[~sel])


# Selected-Q / full-KV control (same section): the selected tokens query every token's
# keys and values at or before their position. Pinned where the two contexts coincide.

def test_fullkv_with_every_token_selected_is_the_sparse_layer():
    w, lw, od, x = _setup()
    bias = I.router_bias(w)
    a = O.layer_fwd(od, O.FULLKV, 1, 0, O.Layer(lw), x, bias=bias)
    b = O.layer_fwd(od, O.SPARSE, 1, 0, O.Layer(lw), x, bias=bias)
    assert np.array_equal(a["y"], b["y"])


def test_fullkv_with_a_selected_prefix_is_the_sparse_layer():
    w, lw, od, x = _setup()
    n = w.T // w.K
    # the first n positions win: their compact order is the position order and every
    # key at or before a selected position is itself selected
    bias = np.where(np.arange(w.T)[None, :] < n, 50.0, -50.0) * np.ones((w.B, 1))
    a = O.layer_fwd(od, O.FULLKV, w.K, 0, O.Layer(lw), x, bias=bias)
    b = O.layer_fwd(od, O.SPARSE, w.K, 0, O.Layer(lw), x, bias=bias)
    assert np.array_equal(a["idx"], np.tile(np.arange(n, dtype=np.int32), (w.B, 1)))
    np.testing.assert_allclose(a["y"], b["y"], rtol=0, atol=1e-12 * np.abs(b["y"]).max())


def test_fullkv_sees_unselected_keys():
    w, lw, od, x = _setup()
    bias = I.router_bias(w)
    a = O.layer_fwd(od, O.FULLKV, w.K, 0, O.Layer(lw), x, bias=bias)
    b = O.layer_fwd(od, O.SPARSE, w.K, 0, O.Layer(lw), x, bias=bias)
    assert np.array_equal(a["idx"], b["idx"])
    assert np.abs(a["y"] - b["y"]).max() > 1e-3
