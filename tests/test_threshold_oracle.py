"""The oracle's causal threshold rule (X-MoD notes, "top-k in training, causal threshold
at evaluation": a token enters when its routing probability is at least 1/2) pinned to
cases with known answers:
  * every logit negative: no token enters, the stream is unchanged bit for bit;
  * every logit overwhelmingly positive with varsigma = 1: every gate is exactly 1, so
    Eq. 7 reduces to the dense layer's x + a + f;
  * exactly T/K logits of each sequence non-negative: the threshold and the top-(T/K)
    rules pick the same tokens, so the two layers agree;
  * the stack under the threshold rule with an overwhelming bias growth: a token that
    entered stays out for the rest of its block."""
import numpy as np

import oracle as O
from oracle import structure as S
from sparse_depth_token_gb300 import inputs as I


def _setup(**over):
    w = I.WORKLOADS["tiny_fp32"].replace(**over)
    lw = I.layer_weights(w, 1)
    od = O.dims(w.B, w.T, w.d, w.hq, w.hkv, w.hd, w.F, w.eps)
    x = I.to_f64(I.residual_stream(w), "fp32")
    return w, lw, od, x


def test_no_logit_non_negative_leaves_the_stream():
    w, lw, od, x = _setup()
    bias = np.full((w.B, w.T), -1e3)
    y, s, mask = O.layer_threshold(od, 0, O.Layer(lw), x, bias=bias)
    assert not mask.any()
    assert np.array_equal(y, x)


def test_all_tokens_with_unit_gate_is_the_dense_layer():
    w, lw, od, x = _setup()
    lw = dict(lw, varsigma=np.float32(1.0))
    bias = np.full((w.B, w.T), 1e3)
    y, s, mask = O.layer_threshold(od, 0, O.Layer(lw), x, bias=bias)
    assert mask.all()
    dense = O.layer_fwd(od, 0, w.K, 0, O.Layer(lw), x)["y"]
    np.testing.assert_allclose(y, dense, rtol=0, atol=1e-12 * np.abs(dense).max())


def test_threshold_equals_topk_when_exactly_n_logits_are_non_negative():
    w, lw, od, x = _setup()
    n = w.T // w.K
    # the logit without bias, then a per-sequence bias that puts the split between
    # the n-th and (n+1)-th largest
    _, s0, _ = O.layer_threshold(od, 0, O.Layer(lw), x, bias=np.zeros((w.B, w.T)))
    srt = -np.sort(-s0, axis=1)
    mid = 0.5 * (srt[:, n - 1] + srt[:, n])
    bias = np.repeat(-mid[:, None], w.T, axis=1)
    y_thr, s, mask = O.layer_threshold(od, 0, O.Layer(lw), x, bias=bias)
    assert np.all(mask.sum(axis=1) == n)
    ref = O.layer_fwd(od, 1, w.K, 0, O.Layer(lw), x, bias=bias)
    sel = np.zeros((w.B, w.T), bool)
    np.put_along_axis(sel, ref["idx"], True, 1)
    assert np.array_equal(sel, mask)
    np.testing.assert_allclose(y_thr, ref["y"], rtol=0, atol=1e-12 * np.abs(ref["y"]).max())


def test_threshold_stack_with_overwhelming_growth_selects_each_token_once_per_block():
    w, lw, od, x = _setup(N1=2, n_layers=11)
    layers = I.all_layer_weights(w)
    kinds = S.schedule(w.N0, w.N1, w.A, w.K)
    big = 1e6
    y, idx, s, mask = O.stack_dyn(od, w.K, 0, kinds, [O.Layer(l) for l in layers], x,
                                  bias=I.router_bias(w), bias_step=big, routing=O.THRESHOLD)
    assert idx is None
    AK = w.K
    for k in range(w.N1):
        blk = mask[k * AK:(k + 1) * AK]
        assert blk.sum(axis=0).max() <= 1                   # at most once per block
        for l in range(1, AK):
            assert not np.any(blk[l] & blk[:l].any(axis=0))
            # penalised tokens are exactly the earlier picks
            assert np.array_equal(s[k * AK + l] < -big / 2, blk[:l].any(axis=0))
        assert np.abs(s[k * AK]).max() < 1e3                # cleared at the anchor
