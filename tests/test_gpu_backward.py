"""GPU parity of the layer backward (xmod_layer_bwd) against the oracle's layer_bwd,
through the C ABI: dx, every weight gradient, dJ/dvarsigma and the Eq. 9 loss, for
sparse layers under Eq. 7 and Eq. 6 (with and without the Eq. 9 term) and dense layers.

Tolerances. fp32 (FFMA kernels throughout): relative 1e-5 as for the forward. bf16:
relative L2 <= 1e-2 (the bound of the bf16 forward); a gradient has no natural unit,
so the max-abs bound 2e-2 is taken relative to the gradient's largest reference entry.
"""
import numpy as np
import pytest

import oracle as O
from sparse_depth_token_gb300 import inputs as I
from tests import _util as U
from tests._gpu import from_dev, need_gpu, oracle_layer, to_dev, torch, xmod_dims, dev_layer

pytestmark = pytest.mark.gpu

GRAD_NAMES = {"w_r": "w_router", "g1": "rms1", "wq": "wq", "wk": "wk", "wv": "wv", "wo": "wo",
              "g2": "rms2", "wg": "w_gate", "wu": "w_up", "wd": "w_down"}


@pytest.fixture(scope="module")
def X():
    need_gpu()
    from sparse_depth_token_gb300 import xmod
    xmod.load()
    return xmod


def _check(got, ref, dtype, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite"
    rl = U.rel_l2(got, ref)
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    mr = float(np.max(np.abs(got - ref))) / scale if scale > 0 else float(np.max(np.abs(got)))
    if dtype == "fp32":
        assert rl <= U.FP32_REL and mr <= U.FP32_REL, f"{what}: rel-L2 {rl:.2e}, max-rel {mr:.2e}"
    else:
        assert rl <= U.BF16_REL_L2 and mr <= U.BF16_MAX_ABS, \
            f"{what}: rel-L2 {rl:.2e}, max-abs/max|ref| {mr:.2e}"


def _run(X, w: I.Workload, kind, gate, route_coef, seed):
    lw = I.layer_weights(w, 0)
    lw["varsigma"] = 0.9
    bias = I.router_bias(w)
    x = I.residual_stream(w)
    if kind == X.LAYER_SPARSE:
        x, _ = U.enforce_routing_margin(x, w.dtype, lw["w_r"], bias, w.K)
    g = np.random.default_rng(seed)
    dyf = g.standard_normal((w.B, w.T, w.d)).astype(np.float32)
    dy = I.f32_to_bf16_bits(dyf) if w.dtype == "bf16" else dyf
    dm = xmod_dims(w)
    ws = torch.zeros(X.bwd_workspace_bytes(dm, w.K), dtype=torch.uint8, device="cuda")
    abi = X.layer_weights(dev_layer(lw, w.dtype), lw["varsigma"])
    xd, dyd = to_dev(x, w.dtype), to_dev(dy, w.dtype)
    dx = torch.empty_like(xd)
    qw, kw = w.hq * w.hd, w.hkv * w.hd
    shapes = {"w_router": (w.d,), "rms1": (w.d,), "wq": (qw, w.d), "wk": (kw, w.d),
              "wv": (kw, w.d), "wo": (w.d, qw), "rms2": (w.d,), "w_gate": (w.F, w.d),
              "w_up": (w.F, w.d), "w_down": (w.d, w.F), "varsigma": (4,), "route_loss": (4,)}
    gd = {k: torch.full(v, float("nan"), dtype=torch.float32, device="cuda")
          for k, v in shapes.items()}
    X.reset_status(ws)
    X.layer_bwd(dm, kind, w.K, gate, abi, xd, torch.from_numpy(bias).cuda()
                if bias is not None else None, dyd, route_coef, dx, X.layer_grads(gd), ws)
    assert X.sync_status(ws) == X.OK
    ref = O.layer_bwd(U_dims(w), kind, w.K, gate, oracle_layer(lw, w.dtype), I.to_f64(x, w.dtype),
                      I.to_f64(dy, w.dtype), bias=bias, route_coef=route_coef)
    _check(from_dev(dx, w.dtype), ref["dx"], w.dtype, "dx")
    for on, an in GRAD_NAMES.items():
        if kind == X.LAYER_DENSE and on == "w_r":
            assert torch.all(gd[an] == 0)
            continue
        _check(gd[an].cpu().numpy(), ref["grads"][on], w.dtype, f"d{on}")
    vs = float(gd["varsigma"][0])
    if kind == X.LAYER_SPARSE and gate == X.GATE_XMOD:
        _check(np.array([vs]), np.array([ref["varsigma"]]), w.dtype, "dvarsigma")
    else:
        assert vs == 0.0
    if kind == X.LAYER_SPARSE:
        _check(np.array([float(gd["route_loss"][0])]), np.array([ref["route_loss"]]), w.dtype,
               "route loss")
    if kind == X.LAYER_SPARSE and route_coef == 0.0:
        # a skipped token's gradient is the upstream gradient, bit for bit
        sel = np.zeros((w.B, w.T), bool)
        np.put_along_axis(sel, ref["idx"], True, 1)
        got = from_dev(dx, w.dtype)
        np.testing.assert_array_equal(got[~sel], I.to_f64(dy, w.dtype)[~sel])


def U_dims(w):
    return O.dims(w.B, w.T, w.d, w.hq, w.hkv, w.hd, w.F, w.eps)


@pytest.mark.parametrize("kind,gate,coef", [(1, 0, 0.0), (1, 1, 0.0), (1, 0, 0.5), (1, 1, 2.0),
                                            (0, 0, 0.0)])
def test_layer_bwd_fp32_tiny(X, kind, gate, coef):
    """The tiny fp32 configuration (d=128, 4/2 heads of 32, F=352, B=2, T=64, K=4)."""
    w = I.WORKLOADS["tiny_fp32"]
    _run(X, w, kind, gate, coef, seed=20 + 3 * kind + gate)


@pytest.mark.parametrize("T,K,kind,gate,coef", [(256, 4, 1, 0, 0.0), (303, 3, 1, 1, 0.0),
                                                (256, 8, 1, 0, 1e-1), (160, 1, 0, 0, 0.0)])
def test_layer_bwd_bf16_tensor_core(X, T, K, kind, gate, coef):
    """bf16, head_dim 128 (tensor-core projections and gradients): A4K8-shaped heads at a
    reduced width, ragged row counts (n = 101: the zero-token padding of the transposed
    operands), both gates, the Eq. 9 term, a dense layer."""
    w = I.WORKLOADS["a4k8_bf16"].replace(B=2, T=T, K=K, d=256, hq=4, hkv=2, F=512, seed=31,
                                         weight_std=0.02 * np.sqrt(1536 / 256))
    _run(X, w, kind, gate, coef, seed=40 + T + K)
