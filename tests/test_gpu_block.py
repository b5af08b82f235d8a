"""GPU parity of the block and of single layers against the CPU oracle, through the C ABI.

Layer outputs are teacher-forced: the oracle runs each layer on the exact input
the GPU layer received. The first sparse layer's inputs are margin-fixed, so
its selection must be bit-exact."""
import numpy as np
import pytest

import oracle as O
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


def _tdt(dtype):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


BLOCK_CASES = {
    # tiny fp32 widths (d=128, 4/2 heads, hd=32, F=352), compact n=16 and a ragged n=37
    "tiny_fp32_n16": I.WORKLOADS["tiny_fp32"].replace(B=2, T=16),
    "tiny_fp32_n37": I.WORKLOADS["tiny_fp32"].replace(B=3, T=37),
    # bf16, hd=128, sizes spanning several 128-row tiles with a ragged tail
    "bf16_hd128_ragged": I.WORKLOADS["a4k8_bf16"].replace(B=2, T=300, d=256, hq=4, hkv=2,
                                                          F=392, seed=21),
    "bf16_gqa3": I.WORKLOADS["a4k8_bf16"].replace(B=1, T=129, d=384, hq=6, hkv=2, F=256, seed=22),
}


@pytest.mark.parametrize("case", sorted(BLOCK_CASES))
@pytest.mark.parametrize("via_idx", [False, True])
def test_block_fwd(X, case, via_idx):
    w = BLOCK_CASES[case]
    n = w.T
    lw = I.layer_weights(w, 0)
    g = np.random.default_rng(3)
    dt = w.dtype
    if via_idx:
        # rows picked from a longer stream through idx
        T_full = 2 * n + 5
        xf = g.standard_normal((w.B, T_full, w.d)).astype(np.float32)
        x = I.f32_to_bf16_bits(xf) if dt == "bf16" else xf
        idx = np.sort(np.stack([g.choice(T_full, n, replace=False) for _ in range(w.B)]), 1)
        idx = idx.astype(np.int32)
        xs = np.stack([x[b, idx[b]] for b in range(w.B)])
        dm = xmod_dims(w, T=T_full)
        src = to_dev(x, dt)
        idx_d = torch.from_numpy(idx).cuda()
    else:
        xf = g.standard_normal((w.B, n, w.d)).astype(np.float32)
        xs = I.f32_to_bf16_bits(xf) if dt == "bf16" else xf
        dm = xmod_dims(w)
        src = to_dev(xs.reshape(w.B * n, w.d), dt)
        idx_d = None
    ws = workspace(dm, dm.T // n)
    a = torch.empty((w.B * n, w.d), dtype=_tdt(dt), device="cuda")
    f = torch.empty_like(a)
    dl = dev_layer(lw, dt)
    X.reset_status(ws)
    X.block_fwd(dm, n, src, idx_d, X.layer_weights(dl, lw["varsigma"]), a, f, ws)
    assert X.sync_status(ws) == X.OK
    od = oracle_dims(w, T=n)
    L = oracle_layer(lw, dt)
    for b in range(w.B):
        a_ref, f_ref = O.block(od, I.to_f64(xs[b], dt), L)
        U.assert_close(from_dev(a[b * n:(b + 1) * n], dt), a_ref, dt, f"a[{b}]")
        U.assert_close(from_dev(f[b * n:(b + 1) * n], dt), f_ref, dt, f"f[{b}]")


# Reduced widths scale the matrix std by sqrt(1536 / d) so that the layer update keeps the
# magnitude it has at the A4K8 width (else it sinks below the bf16 stream's storage precision).
LAYER_CASES = {
    "tiny_fp32": I.WORKLOADS["tiny_fp32"],
    "bf16_small": I.WORKLOADS["a4k8_bf16"].replace(B=2, T=512, d=256, hq=4, hkv=2, F=384, seed=31,
                                                   weight_std=0.049),
    "bf16_ragged_T": I.WORKLOADS["a4k8_bf16"].replace(B=2, T=1000, d=256, hq=6, hkv=2, F=264,
                                                      seed=32, weight_std=0.049),
}


@pytest.mark.parametrize("case", sorted(LAYER_CASES))
@pytest.mark.parametrize("kind,gate", [(1, 0), (1, 1), (0, 0)])
def test_layer_fwd(X, case, kind, gate):
    w = LAYER_CASES[case]
    dt = w.dtype
    K = w.K
    lw = I.layer_weights(w, 1)
    bias = I.router_bias(w)
    x = I.residual_stream(w)
    if kind == 1:
        x, _ = U.enforce_routing_margin(x, dt, lw["w_r"], bias, K)
    dm = xmod_dims(w)
    ws = workspace(dm, K)
    xd = to_dev(x, dt)
    n = w.T // K
    idx = torch.empty((w.B, n), dtype=torch.int32, device="cuda")
    r_sel = torch.empty((w.B, n), dtype=torch.float32, device="cuda")
    X.reset_status(ws)
    X.layer_fwd(dm, kind, K, gate, X.layer_weights(dev_layer(lw, dt), lw["varsigma"]), xd,
                torch.from_numpy(bias).cuda() if bias is not None else None,
                idx if kind == 1 else None, r_sel if kind == 1 else None, ws)
    assert X.sync_status(ws) == X.OK
    ref = O.layer_fwd(oracle_dims(w), kind, K, gate, oracle_layer(lw, dt), I.to_f64(x, dt),
                      bias=bias)
    got = from_dev(xd, dt).reshape(w.B, w.T, w.d)
    x64 = I.to_f64(x, dt)
    if kind == 1:
        np.testing.assert_array_equal(idx.cpu().numpy(), ref["idx"])
        np.testing.assert_allclose(r_sel.cpu().numpy(), ref["r_sel"], rtol=1e-5, atol=1e-6)
        sel = np.zeros((w.B, w.T), bool)
        np.put_along_axis(sel, ref["idx"], True, 1)
        np.testing.assert_array_equal(got[~sel], x64[~sel])   # skip path is bitwise identity
    else:
        sel = np.ones((w.B, w.T), bool)
    U.assert_close(got, ref["y"], dt, "y", stored_ref=got)
    U.assert_close(got[sel] - x64[sel], ref["y"][sel] - x64[sel], dt, "update",
                   stored_ref=got[sel])
