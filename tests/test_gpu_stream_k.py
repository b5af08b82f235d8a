"""Stream-K tensor-core GEMMs (the k-blocks of all tiles split evenly over the CTAs,
a tile cut between two CTAs finished by the one holding its first k-blocks) against
the data-parallel kernels and the oracle.

Stream-K runs when XMOD_STREAM_K=1 asks for it (it measured slower than the
data-parallel tiling on the A4K8 block); here on XMOD_STREAM_K_CTAS CTAs so that tiles
are cut at many places, with pairs switched off so that the gate/up GEMM takes it too."""
import os

import numpy as np
import pytest

import oracle as O
from sparse_depth_token_gb300 import inputs as I
from tests import _util as U
from tests._gpu import dev_layer, from_dev, need_gpu, oracle_dims, oracle_layer, to_dev, torch, workspace, xmod_dims

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def X():
    need_gpu()
    from sparse_depth_token_gb300 import xmod
    xmod.load()
    return xmod


CASES = {
    # M = 1024 dense / 128 sparse rows, q|k|v N = 1024, d = 256, F = 384
    "bf16_small": I.WORKLOADS["a4k8_bf16"].replace(B=2, T=512, d=256, hq=4, hkv=2, F=384,
                                                   seed=51, weight_std=0.049),
    # M = 2000 dense / 250 sparse rows (ragged row tiles), F = 264 (ragged k-blocks)
    "bf16_ragged": I.WORKLOADS["a4k8_bf16"].replace(B=2, T=1000, d=256, hq=6, hkv=2, F=264,
                                                    seed=52, weight_std=0.049),
}


class _Env:
    def __init__(self, **kv):
        self.kv = {k: str(v) for k, v in kv.items()}

    def __enter__(self):
        self.old = {k: os.environ.get(k) for k in self.kv}
        os.environ.update(self.kv)

    def __exit__(self, *exc):
        for k, v in self.old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def _run(X, w, kind, x, lw, bias, **env):
    dt = w.dtype
    dm = xmod_dims(w)
    ws = workspace(dm, w.K)
    xd = to_dev(x, dt)
    with _Env(XMOD_PAIR_MIN_WAVES=999999, **env):
        X.reset_status(ws)
        X.layer_fwd(dm, kind, w.K, 0, X.layer_weights(dev_layer(lw, dt), lw["varsigma"]), xd,
                    torch.from_numpy(bias).cuda() if bias is not None else None, None, None, ws)
        assert X.sync_status(ws) == X.OK
    return xd


def _rel_l2(a, b):
    a = a.float()
    b = b.float()
    return float(torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(b))


@pytest.mark.parametrize("ctas", [3, 7, 13])
@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("kind", [0, 1])
def test_stream_k_matches_data_parallel_and_oracle(X, case, kind, ctas):
    w = CASES[case]
    dt = w.dtype
    lw = I.layer_weights(w, 2)
    bias = I.router_bias(w)
    x = I.residual_stream(w)
    if kind == 1:
        x, _ = U.enforce_routing_margin(x, dt, lw["w_r"], bias, w.K)
    y_sk = _run(X, w, kind, x, lw, bias, XMOD_STREAM_K=1, XMOD_STREAM_K_CTAS=ctas)
    y_dp = _run(X, w, kind, x, lw, bias, XMOD_STREAM_K=0)
    # the same products; only the fp32 sum of a cut tile's two halves is rounded apart
    assert _rel_l2(y_sk, y_dp) < 2e-3
    ref = O.layer_fwd(oracle_dims(w), kind, w.K, 0, oracle_layer(lw, dt), I.to_f64(x, dt),
                      bias=bias)
    got = from_dev(y_sk, dt).reshape(w.B, w.T, w.d)
    U.assert_close(got, ref["y"], dt, "y", stored_ref=got)


def test_stream_k_is_deterministic(X):
    """Cut tiles are summed in one fixed order: repeated runs agree bit for bit."""
    w = CASES["bf16_ragged"]
    lw = I.layer_weights(w, 3)
    bias = I.router_bias(w)
    x = I.residual_stream(w)
    x, _ = U.enforce_routing_margin(x, w.dtype, lw["w_r"], bias, w.K)
    ys = [_run(X, w, 1, x, lw, bias, XMOD_STREAM_K=1, XMOD_STREAM_K_CTAS=11) for _ in range(3)]
    for y in ys[1:]:
        assert torch.equal(y.view(torch.int16), ys[0].view(torch.int16))


def test_stream_k_a4k8_sparse_layer(X):
    """The A4K8 sparse layer at full size (B = 8, T = 4096, d = 1536, 12/4 heads,
    d_ff = 4096: 4096 selected rows), stream-K on all 152 SMs for q|k|v, o-proj and
    down (CTA pairs for gate/up) against data-parallel tiles everywhere."""
    w = I.WORKLOADS["a4k8_bf16"]
    dt = w.dtype
    lw = I.layer_weights(w, 0)
    bias = I.router_bias(w)
    x = I.residual_stream(w)
    dm = xmod_dims(w)
    ws = workspace(dm, w.K)
    outs = []
    for env in ({"XMOD_STREAM_K": 1}, {"XMOD_STREAM_K": 0}):
        xd = to_dev(x, dt)
        with _Env(**env):
            X.reset_status(ws)
            X.layer_fwd(dm, 1, w.K, 0, X.layer_weights(dev_layer(lw, dt), lw["varsigma"]), xd,
                        torch.from_numpy(bias).cuda(), None, None, ws)
            assert X.sync_status(ws) == X.OK
        outs.append(xd)
    assert _rel_l2(outs[0], outs[1]) < 2e-3
    # elementwise: one bf16 rounding step of y (2^-7 of its magnitude) plus the effect
    # of one-step flips in the bf16 intermediates (a, hidden) scaled by the gate
    # varsigma * r <= 1.5: 2^-6 absolute
    a, b = outs[0].float(), outs[1].float()
    excess = (a - b).abs() - (2.0 ** -7 * torch.maximum(a.abs(), b.abs()) + 2.0 ** -6)
    worst = int(torch.argmax(excess))
    assert float(excess.flatten()[worst]) <= 0, (
        worst, float(a.flatten()[worst]), float(b.flatten()[worst]))
