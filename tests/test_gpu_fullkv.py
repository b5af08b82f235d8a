"""GPU: the Selected-Q / full-KV control of X-MoD notes "mechanism controls" -- routed
like a sparse layer, but the selected tokens attend to the keys and values of every
token at or before their position -- against the oracle layer by layer (fp32, and bf16
on the tensor-core path with query positions masking the full-sequence keys), and as
a stack against the layer-by-layer composition bit for bit."""
import numpy as np
import pytest

import oracle as O
from oracle import structure as S
from sparse_depth_token_gb300 import inputs as I
from tests import _util as U
from tests._gpu import (dev_layer, from_dev, need_gpu, oracle_dims, oracle_layer, to_dev, torch,
                        workspace, xmod_dims)

pytestmark = pytest.mark.gpu

FULLKV = 4


@pytest.fixture(scope="module")
def X():
    need_gpu()
    from sparse_depth_token_gb300 import xmod
    xmod.load()
    return xmod


CASES = {
    "tiny_fp32": I.WORKLOADS["tiny_fp32"],
    # n = 64 queries over 512 keys; and T = 1000 (n = 125, keys off every tile edge)
    "bf16_small": I.WORKLOADS["a4k8_bf16"].replace(B=2, T=512, d=256, hq=4, hkv=2, F=384,
                                                   seed=91, weight_std=0.049),
    "bf16_ragged": I.WORKLOADS["a4k8_bf16"].replace(B=2, T=1000, d=256, hq=6, hkv=2, F=264,
                                                    seed=92, weight_std=0.049),
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("gate", [0, 1])
def test_fullkv_layer_against_oracle(X, case, gate):
    w = CASES[case]
    dt = w.dtype
    lw = I.layer_weights(w, 5)
    bias = I.router_bias(w)
    x = I.residual_stream(w)
    x, _ = U.enforce_routing_margin(x, dt, lw["w_r"], bias, w.K)
    dm = xmod_dims(w)
    ws = workspace(dm, w.K)
    xd = to_dev(x, dt)
    X.reset_status(ws)
    X.layer_fwd(dm, FULLKV, w.K, gate, X.layer_weights(dev_layer(lw, dt), lw["varsigma"]), xd,
                torch.from_numpy(bias).cuda() if bias is not None else None, None, None, ws)
    assert X.sync_status(ws) == X.OK
    ref = O.layer_fwd(oracle_dims(w), O.FULLKV, w.K, gate, oracle_layer(lw, dt), I.to_f64(x, dt),
                      bias=bias)
    got = from_dev(xd, dt).reshape(w.B, w.T, w.d)
    x64 = I.to_f64(x, dt)
    sel = np.zeros((w.B, w.T), bool)
    np.put_along_axis(sel, ref["idx"], True, 1)
    np.testing.assert_array_equal(got[~sel], x64[~sel])
    U.assert_close(got, ref["y"], dt, "y", stored_ref=got)
    U.assert_close(got[sel] - x64[sel], ref["y"][sel] - x64[sel], dt, "update",
                   stored_ref=got[sel])


def test_fullkv_stack_is_the_layer_composition(X):
    w = CASES["bf16_small"].replace(A=1, n_layers=9)
    kinds = [FULLKV] * 8 + [S.DENSE]
    layers = I.all_layer_weights(w, len(kinds))
    bias = I.router_bias(w)
    x = I.residual_stream(w)
    x, _ = U.enforce_routing_margin(x, w.dtype, layers[0]["w_r"], bias, w.K)
    abi = [X.layer_weights(dev_layer(l, w.dtype), l["varsigma"]) for l in layers]
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
