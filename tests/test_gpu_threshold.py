"""GPU: the causal threshold rule (X-MoD notes, "top-k in training, causal threshold at
evaluation": a token enters when r = sigmoid(s) >= 1/2) against the oracle.

Sequences take different numbers of tokens -- few, many, none -- so the block runs
on a variable number of rows per sequence (row counts known only on the device). Tokens
whose logit lies within 1e-3 of 0 have their bias pushed out of that band first (the
bias is a free input), so the GPU's fp32 logits and the oracle's double logits decide
alike. The stack under the threshold rule equals the layer-by-layer composition bit
for bit, and its statistics are those of the rule."""
import numpy as np
import pytest

import oracle as O
from oracle import structure as S
from sparse_depth_token_gb300 import inputs as I
from tests import _util as U
from tests._gpu import (dev_layer, from_dev, need_gpu, oracle_dims, oracle_layer, to_dev, torch,
                        workspace, xmod_dims)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def X():
    need_gpu()
    from sparse_depth_token_gb300 import xmod
    xmod.load()
    return xmod


CASES = {
    # B = 3: about 20% of the tokens, about 70%, none
    "bf16_small": I.WORKLOADS["a4k8_bf16"].replace(B=3, T=512, d=256, hq=4, hkv=2, F=384,
                                                   seed=61, weight_std=0.049),
    # T = 1000: row counts off every tile boundary
    "bf16_ragged": I.WORKLOADS["a4k8_bf16"].replace(B=2, T=1000, d=256, hq=6, hkv=2, F=264,
                                                    seed=62, weight_std=0.049),
}
OFFSETS = (-0.8, 0.5, -1e3)


def _bias_with_margin(w, x, w_r, margin=1e-3):
    """Per-sequence offsets plus the workload's token bias, with every logit moved at
    least `margin` away from 0 (oracle logits on the stored inputs)."""
    bias = I.router_bias(w).astype(np.float64)
    bias += np.array([OFFSETS[b % len(OFFSETS)] for b in range(w.B)])[:, None]
    s, _ = O.router(I.to_f64(x, w.dtype), I.to_f64(w_r, w.dtype), bias=bias)
    near = np.abs(s) < margin
    bias[near] += np.where(s[near] >= 0, 2 * margin, -2 * margin)
    return bias.astype(np.float32)


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("gate", [0, 1])
def test_threshold_layer_against_oracle(X, case, gate):
    w = CASES[case]
    dt = w.dtype
    lw = I.layer_weights(w, 3)
    x = I.residual_stream(w)
    bias = _bias_with_margin(w, x, lw["w_r"])
    dm = xmod_dims(w)
    ws = workspace(dm, w.K)
    xd = to_dev(x, dt)
    counts = torch.full((w.B,), -1, dtype=torch.int32, device="cuda")
    X.reset_status(ws)
    X.layer_fwd_threshold(dm, gate, X.layer_weights(dev_layer(lw, dt), lw["varsigma"]), xd,
                          torch.from_numpy(bias).cuda(), ws, count_out=counts)
    assert X.sync_status(ws) == X.OK
    y, s, mask = O.layer_threshold(oracle_dims(w), gate, oracle_layer(lw, dt), I.to_f64(x, dt),
                                   bias=bias.astype(np.float64))
    assert np.array_equal(counts.cpu().numpy(), mask.sum(axis=1))
    if w.B >= 3:
        assert mask[2].sum() == 0 and 0 < mask[0].sum() < mask[1].sum()
    got = from_dev(xd, dt).reshape(w.B, w.T, w.d)
    x64 = I.to_f64(x, dt)
    np.testing.assert_array_equal(got[~mask], x64[~mask])      # skipped rows: identity
    U.assert_close(got, y, dt, "y", stored_ref=got)
    U.assert_close(got[mask] - x64[mask], y[mask] - x64[mask], dt, "update", stored_ref=got[mask])


def _stack_setup(X, w):
    layers = I.all_layer_weights(w)
    kinds = S.schedule(w.N0, w.N1, w.A, w.K)
    x = I.residual_stream(w)
    first = kinds.index(S.SPARSE)
    bias = _bias_with_margin(w, x, layers[first]["w_r"])
    abi = [X.layer_weights(dev_layer(l, w.dtype), l["varsigma"]) for l in layers]
    return layers, kinds, x, bias, abi


def test_threshold_stack_is_the_layer_composition(X):
    # [S] x 8 + [D] at A4K8 widths
    w = I.WORKLOADS["a4k8_bf16"].replace(B=3, T=512, d=256, hq=4, hkv=2, F=384, A=1,
                                         n_layers=9, seed=63, weight_std=0.049)
    layers, kinds, x, bias, abi = _stack_setup(X, w)
    dm = xmod_dims(w)
    ws = workspace(dm, w.K)
    bd = torch.from_numpy(bias).cuda()
    # layer by layer
    xl = to_dev(x, w.dtype)
    X.reset_status(ws)
    per_layer = []
    for l, k in enumerate(kinds):
        if k == S.SPARSE:
            cnt = torch.zeros((w.B,), dtype=torch.int32, device="cuda")
            X.layer_fwd_threshold(dm, w.gate, abi[l], xl, bd, ws, count_out=cnt)
            per_layer.append(cnt)
        else:
            X.layer_fwd(dm, 0, w.K, w.gate, abi[l], xl, bd, None, None, ws)
    assert X.sync_status(ws) == X.OK
    # the stack
    xs = to_dev(x, w.dtype)
    n_sparse = kinds.count(S.SPARSE)
    st = torch.full((n_sparse, w.B, 4), -1, dtype=torch.int32, device="cuda")
    uh = torch.full((w.N1, w.B, w.K + 1), -1, dtype=torch.int32, device="cuda")
    X.reset_status(ws)
    X.stack_fwd_ex(dm, w.K, w.A, w.N0, w.N1, w.gate, abi, xs, bd, ws, layer_stats=st,
                   update_hist=uh, routing=X.ROUTE_THRESHOLD)
    assert X.sync_status(ws) == X.OK
    assert torch.equal(xs.view(torch.int16), xl.view(torch.int16))
    st = st.cpu().numpy()
    counts = torch.stack(per_layer).cpu().numpy()
    assert np.array_equal(st[:, :, 0], counts) and np.array_equal(st[:, :, 1], counts)
    assert np.all(st[:, :, 2] == w.T)
    assert np.all(uh.cpu().numpy().sum(axis=2) == w.T)
    assert counts[:, 2].max() == 0 and counts[:, 1].min() > 0


def test_threshold_stack_overwhelming_growth(X):
    w = I.WORKLOADS["a4k8_bf16"].replace(B=2, T=512, d=256, hq=4, hkv=2, F=384, A=1,
                                         n_layers=9, seed=64, weight_std=0.049)
    layers, kinds, x, bias, abi = _stack_setup(X, w)
    dm = xmod_dims(w)
    ws = workspace(dm, w.K)
    xs = to_dev(x, w.dtype)
    st = torch.full((8, w.B, 4), -1, dtype=torch.int32, device="cuda")
    uh = torch.full((1, w.B, w.K + 1), -1, dtype=torch.int32, device="cuda")
    X.reset_status(ws)
    X.stack_fwd_ex(dm, w.K, w.A, w.N0, w.N1, w.gate, abi, xs, torch.from_numpy(bias).cuda(), ws,
                   bias_step=1e4, layer_stats=st, update_hist=uh, routing=X.ROUTE_THRESHOLD)
    assert X.sync_status(ws) == X.OK
    st, uh = st.cpu().numpy(), uh.cpu().numpy()
    assert np.all(st[:, :, 3] == 0)            # no token enters twice in the block
    assert np.all(uh[:, :, 2:] == 0)
    assert np.array_equal(uh[0, :, 1], st[:, :, 0].sum(axis=0))
