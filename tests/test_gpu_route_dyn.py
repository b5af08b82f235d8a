"""GPU: the stack with token-choice bias dynamics and routing statistics
(xmod_stack_fwd_ex) against the oracle and the closed-form rotation.

X-MoD notes, Eq. 8 and the paragraph after it (a token's bias grows with each
selection inside a sparse-dense block and clears at the dense anchor) and Table 10's
diagnostics. The tiny fp32 stack runs end to end against the oracle, statistics
included (counted plainly from the oracle's selections and logits). The bf16 A4K8
widths run the tensor-core path: no growth equals xmod_stack_fwd bit for bit, asking
for statistics changes no result, and an overwhelming growth gives the closed-form
rotation (every token updated exactly once per block of K sparse layers)."""
import numpy as np
import pytest

import oracle as O
from oracle import diagnostics as D
from oracle import structure as S
from sparse_depth_token_gb300 import diagnostics as PD
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


def _setup(X, w):
    layers = I.all_layer_weights(w)
    kinds = S.schedule(w.N0, w.N1, w.A, w.K)
    bias = I.router_bias(w)
    x = I.residual_stream(w)
    first = kinds.index(S.SPARSE)
    x, _ = U.enforce_routing_margin(x, w.dtype, layers[first]["w_r"], bias, w.K)
    abi = [X.layer_weights(dev_layer(l, w.dtype), l["varsigma"]) for l in layers]
    return layers, kinds, bias, x, abi


def _run(X, w, kinds, x, bias, abi, bias_step, stats=True, ex=True):
    dm = xmod_dims(w)
    ws = workspace(dm, w.K)
    xd = to_dev(x, w.dtype)
    bd = torch.from_numpy(bias).cuda() if bias is not None else None
    AK = round(w.A * w.K)
    n_sparse = kinds.count(S.SPARSE)
    st = torch.full((n_sparse, w.B, 4), -1, dtype=torch.int32, device="cuda") if stats else None
    uh = torch.full((w.N1, w.B, AK + 1), -1, dtype=torch.int32, device="cuda") if stats else None
    X.reset_status(ws)
    if ex:
        X.stack_fwd_ex(dm, w.K, w.A, w.N0, w.N1, w.gate, abi, xd, bd, ws, bias_step=bias_step,
                       layer_stats=st, update_hist=uh)
    else:
        X.stack_fwd(dm, w.K, w.A, w.N0, w.N1, w.gate, abi, xd, bd, ws)
    assert X.sync_status(ws) == X.OK
    return xd, (st.cpu().numpy() if stats else None), (uh.cpu().numpy() if stats else None)


@pytest.mark.parametrize("bias_step", [0.3, 1e4])
def test_tiny_fp32_dynamics_end_to_end(X, bias_step):
    # [D] + ([S(4)] x 4 + [D]) x 2
    w = I.WORKLOADS["tiny_fp32"].replace(N1=2, n_layers=11)
    layers, kinds, bias, x, abi = _setup(X, w)
    xd, st, uh = _run(X, w, kinds, x, bias, abi, bias_step)
    ref, idx, s, _ = O.stack_dyn(oracle_dims(w), w.K, w.gate, kinds,
                              [oracle_layer(l, "fp32") for l in layers], I.to_f64(x, "fp32"),
                              bias=bias, bias_step=bias_step)
    U.assert_close(from_dev(xd, "fp32").reshape(ref.shape), ref, "fp32", "stack")
    AK = w.K
    masks = D.masks_from_idx(idx, w.T)
    thr = s >= 0
    assert np.all(st[:, :, 0] == w.T // w.K)
    assert np.array_equal(st[:, :, 1], thr.sum(2))
    assert np.array_equal(st[:, :, 2], (masks == thr).sum(2))
    for l in range(len(idx)):
        want = np.logical_and(masks[l], masks[l - 1]).sum(1) if l % AK else 0
        assert np.all(st[l, :, 3] == want)
    for k in range(w.N1):
        c = masks[k * AK:(k + 1) * AK].sum(0)
        for b in range(w.B):
            assert np.array_equal(uh[k, b], np.bincount(c[b], minlength=AK + 1))
    if bias_step > 1e3:   # the closed-form rotation
        diag = PD.route_diagnostics(st, uh, w.T, AK)
        assert diag.coverage == 1.0 and diag.jaccard == 0.0
        assert diag.update_dist[1] == 1.0


def test_bf16_dynamics_tensor_core_path(X):
    # A4K8 widths, two blocks of K = 8 sparse layers: [S(8)] x 8 + [D], twice
    w = I.WORKLOADS["a4k8_bf16"].replace(B=2, T=512, d=256, hq=4, hkv=2, F=384, A=1, N1=2,
                                         n_layers=18, weight_std=0.049, seed=51)
    layers, kinds, bias, x, abi = _setup(X, w)
    plain, _, _ = _run(X, w, kinds, x, bias, abi, 0.0, stats=False, ex=False)
    same, st0, uh0 = _run(X, w, kinds, x, bias, abi, 0.0)
    assert torch.equal(plain.view(torch.int16), same.view(torch.int16))
    assert np.all(st0[:, :, 0] == w.T // w.K) and np.all(uh0.sum(2) == w.T)
    rot, st, uh = _run(X, w, kinds, x, bias, abi, 1e4)
    rot2, _, _ = _run(X, w, kinds, x, bias, abi, 1e4, stats=False)
    assert torch.equal(rot.view(torch.int16), rot2.view(torch.int16))
    assert np.all(st[:, :, 0] == w.T // w.K)
    assert np.all(st[:, :, 3] == 0)                      # no token twice in a block
    expect = np.zeros(w.K + 1, np.int64)
    expect[1] = w.T
    assert np.all(uh == expect)                          # every token exactly once
    # agreement counts both rules' joint picks and joint skips: |agree| = T - |sel xor thr|,
    # which lies between T - |sel| - |thr| and T - ||sel| - |thr||
    lo = w.T - st[:, :, 0] - st[:, :, 1]
    hi = w.T - np.abs(st[:, :, 0] - st[:, :, 1])
    assert np.all((st[:, :, 2] >= lo) & (st[:, :, 2] <= hi))
