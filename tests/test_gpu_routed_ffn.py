"""GPU: the Routed-FFN control of X-MoD notes "mechanism controls" -- full-sequence
attention layers (ATTN: x += a on every token) and FFN-only refinements of the
top-(T/K) tokens (ROUTED_FFN: a = 0 in the gated residual) -- against the oracle, layer
by layer and as the stack ([Dense] + ([FullAttn] + [Routed-FFN] x K) x A + [Dense]),
the stack also against the layer-by-layer composition bit for bit, with an
overwhelming bias growth giving the closed-form rotation over the block."""
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
    "tiny_fp32": I.WORKLOADS["tiny_fp32"],
    "bf16_small": I.WORKLOADS["a4k8_bf16"].replace(B=2, T=512, d=256, hq=4, hkv=2, F=384,
                                                   seed=81, weight_std=0.049),
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("kind,gate", [(S.ATTN, 0), (S.RFFN, 0), (S.RFFN, 1)])
def test_variant_layer_against_oracle(X, case, kind, gate):
    w = CASES[case]
    if kind == S.ATTN and w.dtype == "bf16":
        # the attention half alone moves the stream less than the whole block: a 1.25x
        # matrix scale (about 1.6x on a = o Wo^T) keeps its update above the bf16
        # stream's storage rounding, as the block tests scale reduced widths
        w = w.replace(weight_std=1.25 * w.weight_std)
    dt = w.dtype
    lw = I.layer_weights(w, 4)
    bias = I.router_bias(w)
    x = I.residual_stream(w)
    if kind == S.RFFN:
        x, _ = U.enforce_routing_margin(x, dt, lw["w_r"], bias, w.K)
    dm = xmod_dims(w)
    ws = workspace(dm, w.K)
    xd = to_dev(x, dt)
    X.reset_status(ws)
    X.layer_fwd(dm, kind, w.K, gate, X.layer_weights(dev_layer(lw, dt), lw["varsigma"]), xd,
                torch.from_numpy(bias).cuda() if bias is not None else None, None, None, ws)
    assert X.sync_status(ws) == X.OK
    ref = O.layer_fwd(oracle_dims(w), kind, w.K, gate, oracle_layer(lw, dt), I.to_f64(x, dt),
                      bias=bias)
    got = from_dev(xd, dt).reshape(w.B, w.T, w.d)
    x64 = I.to_f64(x, dt)
    if kind == S.RFFN:
        sel = np.zeros((w.B, w.T), bool)
        np.put_along_axis(sel, ref["idx"], True, 1)
        np.testing.assert_array_equal(got[~sel], x64[~sel])
    else:
        sel = np.ones((w.B, w.T), bool)
    U.assert_close(got, ref["y"], dt, "y", stored_ref=got)
    U.assert_close(got[sel] - x64[sel], ref["y"][sel] - x64[sel], dt, "update",
                   stored_ref=got[sel])


def _kinds(K):
    # [Dense] + (([FullAttn] + [Routed-FFN] x K) x 2 + [Dense])
    return S.schedule_routed_ffn(1, [(2 * K, 1)], K)


def _stack_setup(X, w, kinds):
    layers = I.all_layer_weights(w, len(kinds))
    bias = I.router_bias(w)
    x = I.residual_stream(w)
    first = kinds.index(S.RFFN)
    x, _ = U.enforce_routing_margin(x, w.dtype, layers[first]["w_r"], bias, w.K)
    abi = [X.layer_weights(dev_layer(l, w.dtype), l["varsigma"]) for l in layers]
    return layers, bias, x, abi


def test_routed_ffn_stack_fp32_against_oracle(X):
    w = I.WORKLOADS["tiny_fp32"]
    kinds = _kinds(w.K)
    layers, bias, x, abi = _stack_setup(X, w, kinds)
    dm = xmod_dims(w)
    ws = workspace(dm, w.K)
    xd = to_dev(x, "fp32")
    X.reset_status(ws)
    X.stack_fwd_sched(dm, w.K, kinds, w.gate, abi, xd, torch.from_numpy(bias).cuda(), ws)
    assert X.sync_status(ws) == X.OK
    ref = O.stack_fwd(oracle_dims(w), w.K, w.gate, kinds,
                      [oracle_layer(l, "fp32") for l in layers], I.to_f64(x, "fp32"), bias=bias)
    U.assert_close(from_dev(xd, "fp32").reshape(ref.shape), ref, "fp32", "stack")


def test_routed_ffn_stack_bf16_composition_and_rotation(X):
    w = CASES["bf16_small"]
    kinds = _kinds(w.K)
    layers, bias, x, abi = _stack_setup(X, w, kinds)
    dm = xmod_dims(w)
    ws = workspace(dm, w.K)
    bd = torch.from_numpy(bias).cuda()
    xl = to_dev(x, w.dtype)
    X.reset_status(ws)
    for l, k in enumerate(kinds):
        X.layer_fwd(dm, k, w.K, w.gate, abi[l], xl, bd, None, None, ws)
    xs = to_dev(x, w.dtype)
    X.stack_fwd_sched(dm, w.K, kinds, w.gate, abi, xs, bd, ws)
    assert X.sync_status(ws) == X.OK
    assert torch.equal(xs.view(torch.int16), xl.view(torch.int16))
    # 2K routed layers in one block, each taking T / K: every token exactly twice
    n_routed = kinds.count(S.RFFN)
    st = torch.full((n_routed, w.B, 4), -1, dtype=torch.int32, device="cuda")
    uh = torch.full((1, w.B, n_routed + 1), -1, dtype=torch.int32, device="cuda")
    xr = to_dev(x, w.dtype)
    X.stack_fwd_sched(dm, w.K, kinds, w.gate, abi, xr, bd, ws, bias_step=1e4, layer_stats=st,
                      update_hist=uh)
    assert X.sync_status(ws) == X.OK
    uh = uh.cpu().numpy()
    expect = np.zeros(n_routed + 1, np.int64)
    expect[2] = w.T
    assert np.all(uh[0] == expect)
    st = st.cpu().numpy()
    assert np.all(st[:, :, 0] == w.T // w.K)
    assert np.all(st[1:w.K, :, 3] == 0)      # no repeat inside the first K layers
