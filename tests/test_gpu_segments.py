"""GPU: stacks in an explicit layer order -- the heterogeneous segment stacks of X-MoD
notes Eq. 35 / Eq. 36 (a shorter first sparse segment, then longer ones) -- through
xmod_stack_fwd_sched, against the oracle end to end (fp32) and against the
layer-by-layer composition bit for bit (bf16 tensor-core path, statistics included)."""
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


# [Dense] + ([Sparse] x 2 + [Dense]) + ([Sparse] x 3 + [Dense]): Eq. 35's shape, shortened
def _kinds():
    return S.schedule_segments(1, [(2, 1), (3, 1)])


def _setup(X, w, kinds):
    layers = I.all_layer_weights(w, len(kinds))
    bias = I.router_bias(w)
    x = I.residual_stream(w)
    first = kinds.index(S.SPARSE)
    x, _ = U.enforce_routing_margin(x, w.dtype, layers[first]["w_r"], bias, w.K)
    abi = [X.layer_weights(dev_layer(l, w.dtype), l["varsigma"]) for l in layers]
    return layers, bias, x, abi


def test_schedule_shape():
    k = _kinds()
    assert k == [S.DENSE, S.SPARSE, S.SPARSE, S.DENSE, S.SPARSE, S.SPARSE, S.SPARSE, S.DENSE]


def test_segment_stack_fp32_against_oracle(X):
    w = I.WORKLOADS["tiny_fp32"]
    kinds = _kinds()
    layers, bias, x, abi = _setup(X, w, kinds)
    dm = xmod_dims(w)
    ws = workspace(dm, w.K)
    xd = to_dev(x, "fp32")
    X.reset_status(ws)
    X.stack_fwd_sched(dm, w.K, kinds, w.gate, abi, xd, torch.from_numpy(bias).cuda(), ws)
    assert X.sync_status(ws) == X.OK
    ref = O.stack_fwd(oracle_dims(w), w.K, w.gate, kinds,
                      [oracle_layer(l, "fp32") for l in layers], I.to_f64(x, "fp32"), bias=bias)
    U.assert_close(from_dev(xd, "fp32").reshape(ref.shape), ref, "fp32", "stack")


def test_segment_stack_bf16_is_the_layer_composition(X):
    w = I.WORKLOADS["a4k8_bf16"].replace(B=2, T=512, d=256, hq=4, hkv=2, F=384, seed=71,
                                         weight_std=0.049)
    kinds = _kinds()
    layers, bias, x, abi = _setup(X, w, kinds)
    dm = xmod_dims(w)
    ws = workspace(dm, w.K)
    bd = torch.from_numpy(bias).cuda()
    xl = to_dev(x, w.dtype)
    X.reset_status(ws)
    for l, k in enumerate(kinds):
        X.layer_fwd(dm, 1 if k == S.SPARSE else 0, w.K, w.gate, abi[l], xl, bd, None, None, ws)
    xs = to_dev(x, w.dtype)
    st = torch.full((5, w.B, 4), -1, dtype=torch.int32, device="cuda")
    uh = torch.full((2, w.B, 4), -1, dtype=torch.int32, device="cuda")   # 2 blocks, L_max = 3
    X.stack_fwd_sched(dm, w.K, kinds, w.gate, abi, xs, bd, ws, layer_stats=st, update_hist=uh)
    assert X.sync_status(ws) == X.OK
    assert torch.equal(xs.view(torch.int16), xl.view(torch.int16))
    st, uh = st.cpu().numpy(), uh.cpu().numpy()
    n = w.T // w.K
    assert np.all(st[:, :, 0] == n)
    assert np.all(uh.sum(axis=2) == w.T)
    assert np.all(uh[0, :, 3] == 0)                  # the 2-layer block updates at most twice
    assert np.all((uh[0] * np.arange(4)).sum(axis=1) == 2 * n)
    assert np.all((uh[1] * np.arange(4)).sum(axis=1) == 3 * n)
