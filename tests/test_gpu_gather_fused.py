"""The gathered RMSNorm inside the q|k|v GEMM's operand load (XMOD_GATHER_FUSED=1: TMA
gather4 of the selected stream rows, the RMSNorm gain applied in shared memory and
1 / rms in the epilogue) against the oracle, on a sparse layer (top-(T/K) selection,
ragged row tiles) and on the block entry point with positions (idx); the default path
(a gathered, normalised copy) meets the same bar on the same inputs and selects the
same tokens."""
import os

import numpy as np
import pytest

import oracle as O
from sparse_depth_token_gb300 import inputs as I
from tests import _util as U
from tests._gpu import dev_layer, from_dev, need_gpu, oracle_dims, oracle_layer, to_dev, torch, workspace, xmod_dims

pytestmark = pytest.mark.gpu

CASES = {
    # n = 62 selected of T = 500 per sequence (K = 8): one ragged row tile per layer
    "ragged": I.WORKLOADS["a4k8_bf16"].replace(B=2, T=500, d=320, hq=4, hkv=2, F=384, seed=71,
                                               weight_std=0.049),
    # n = 256 of 2048: two full row tiles per sequence, d spanning five k-blocks
    "tiles": I.WORKLOADS["a4k8_bf16"].replace(B=2, T=2048, d=320, hq=4, hkv=2, F=256, seed=72,
                                              weight_std=0.049),
}


@pytest.fixture(scope="module")
def X():
    need_gpu()
    from sparse_depth_token_gb300 import xmod
    xmod.load()
    return xmod


def _with_fused(on, fn):
    old = os.environ.get("XMOD_GATHER_FUSED")
    os.environ["XMOD_GATHER_FUSED"] = "1" if on else "0"
    try:
        return fn()
    finally:
        if old is None:
            del os.environ["XMOD_GATHER_FUSED"]
        else:
            os.environ["XMOD_GATHER_FUSED"] = old


@pytest.mark.parametrize("case", sorted(CASES))
def test_sparse_layer_with_fused_gather(X, case):
    w = CASES[case]
    lw = I.layer_weights(w, 1)
    lw["g1"] = I.f32_to_bf16_bits((1.0 + 0.25 * np.random.default_rng(3).standard_normal(w.d))
                                  .astype(np.float32))   # a live RMSNorm gain
    bias = I.router_bias(w)
    x, _ = U.enforce_routing_margin(I.residual_stream(w), "bf16", lw["w_r"], bias, w.K)
    dm = xmod_dims(w)
    ws = workspace(dm, w.K)
    n = w.T // w.K
    abi = X.layer_weights(dev_layer(lw, "bf16"), lw["varsigma"])

    def run():
        xd = to_dev(x, "bf16")
        idx = torch.empty((w.B, n), dtype=torch.int32, device="cuda")
        X.reset_status(ws)
        X.layer_fwd(dm, 1, w.K, 0, abi, xd, torch.from_numpy(bias).cuda(), idx, None, ws)
        assert X.sync_status(ws) == X.OK
        return from_dev(xd, "bf16").reshape(w.B, w.T, w.d), idx.cpu().numpy()

    got, idx = _with_fused(True, run)
    base, idx0 = _with_fused(False, run)
    np.testing.assert_array_equal(idx, idx0)
    ref = O.layer_fwd(oracle_dims(w), 1, w.K, 0, oracle_layer(lw, "bf16"), I.to_f64(x, "bf16"),
                      bias=bias)
    np.testing.assert_array_equal(idx, ref["idx"])
    U.assert_close(got, ref["y"], "bf16", "fused layer y", stored_ref=got)
    U.assert_close(base, ref["y"], "bf16", "default layer y", stored_ref=base)


def test_block_fwd_with_fused_gather(X):
    w = CASES["ragged"]
    lw = I.layer_weights(w, 2)
    g = np.random.default_rng(4)
    n = w.T // w.K
    idx = np.sort(np.stack([g.choice(w.T, n, replace=False) for _ in range(w.B)]), 1)
    idx = idx.astype(np.int32)
    x = I.residual_stream(w)
    dm = xmod_dims(w)
    ws = workspace(dm, w.K)
    abi = X.layer_weights(dev_layer(lw, "bf16"), lw["varsigma"])
    xd = to_dev(x, "bf16")
    idx_d = torch.from_numpy(idx).cuda()

    def run():
        a = torch.empty((w.B * n, w.d), dtype=torch.bfloat16, device="cuda")
        f = torch.empty_like(a)
        X.reset_status(ws)
        X.block_fwd(dm, n, xd, idx_d, abi, a, f, ws)
        assert X.sync_status(ws) == X.OK
        return from_dev(a, "bf16"), from_dev(f, "bf16")

    a, f = _with_fused(True, run)
    od = oracle_dims(w, B=1, T=n)
    L = oracle_layer(lw, "bf16")
    x64 = I.to_f64(x, "bf16")
    for b in range(w.B):
        ra, rf = O.block(od, x64[b, idx[b]], L)
        U.assert_close(a[b * n:(b + 1) * n], ra, "bf16", f"a[{b}]")
        U.assert_close(f[b * n:(b + 1) * n], rf, "bf16", f"f[{b}]")
