"""The CTA-pair GEMM kernels (tcgen05 cta_group::2, 256 x 256 tiles) against the
single-CTA kernels and the oracle.

The library puts a GEMM on CTA pairs from six waves of pair tiles up (about 450 tiles),
or below that when its waves-times-width estimate favours them clearly; at test sizes
this test forces them (XMOD_PAIR_MIN_WAVES=0) or keeps them off (a huge threshold).
Single layers (dense and sparse) run once each way: the q|k|v, o-projection, gate/up
and down-projection epilogues all run on pairs, with ragged row and column tiles."""
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
    # M = 1024 dense rows: 4 pair rows of tiles; q|k|v N = 1024, d = 256, F = 384
    "bf16_small": I.WORKLOADS["a4k8_bf16"].replace(B=2, T=512, d=256, hq=4, hkv=2, F=384,
                                                   seed=41, weight_std=0.049),
    # M = 2000 dense / 250 sparse rows (the last pair tile half empty), F = 264 (ragged)
    "bf16_ragged": I.WORKLOADS["a4k8_bf16"].replace(B=2, T=1000, d=256, hq=6, hkv=2, F=264,
                                                    seed=42, weight_std=0.049),
}


def _run(X, w, kind, x, lw, bias, pairs, pair_bn=None):
    dt = w.dtype
    dm = xmod_dims(w)
    ws = workspace(dm, w.K)
    xd = to_dev(x, dt)
    env = {"XMOD_PAIR_MIN_WAVES": "0" if pairs else "999999",
           "XMOD_STREAM_K": "0",   # data-parallel single-CTA tiles: the same k order
           "XMOD_PAIR_BN": str(pair_bn) if pair_bn else None}
    old = {k: os.environ.get(k) for k in env}
    for k, v in env.items():
        if v is None:
            os.environ.pop(k, None)
        else:
            os.environ[k] = v
    try:
        X.reset_status(ws)
        X.layer_fwd(dm, kind, w.K, 0, X.layer_weights(dev_layer(lw, dt), lw["varsigma"]), xd,
                    torch.from_numpy(bias).cuda() if bias is not None else None, None, None, ws)
        assert X.sync_status(ws) == X.OK
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return xd


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("kind", [0, 1])
def test_pair_gemms_match_single_cta_and_oracle(X, case, kind):
    w = CASES[case]
    dt = w.dtype
    lw = I.layer_weights(w, 2)
    bias = I.router_bias(w)
    x = I.residual_stream(w)
    if kind == 1:
        x, _ = U.enforce_routing_margin(x, dt, lw["w_r"], bias, w.K)
    y_pair = _run(X, w, kind, x, lw, bias, pairs=True)
    y_single = _run(X, w, kind, x, lw, bias, pairs=False)
    # each output element is the same dot product in the same k order either way
    assert torch.equal(y_pair.view(torch.int16), y_single.view(torch.int16))
    ref = O.layer_fwd(oracle_dims(w), kind, w.K, 0, oracle_layer(lw, dt), I.to_f64(x, dt),
                      bias=bias)
    got = from_dev(y_pair, dt).reshape(w.B, w.T, w.d)
    U.assert_close(got, ref["y"], dt, "y", stored_ref=got)


CASES_192 = {
    # d = 384: the o-projection and down GEMMs two 256 x 192 pair tiles wide (q|k|v,
    # whose q / k / v boundaries fall off the 192 grid, stays on 256-wide pairs)
    "bf16_d384": I.WORKLOADS["a4k8_bf16"].replace(B=2, T=512, K=4, d=384, hq=3, hkv=1, F=384,
                                                  seed=43, weight_std=0.049),
    # d = 320: the second column tile is ragged (128 of its 192 columns exist)
    "bf16_d320": I.WORKLOADS["a4k8_bf16"].replace(B=2, T=512, K=4, d=320, hq=2, hkv=1, F=264,
                                                  seed=44, weight_std=0.049),
}


@pytest.mark.parametrize("case", sorted(CASES_192))
@pytest.mark.parametrize("kind", [0, 1])
def test_pair_tiles_192_wide(X, case, kind):
    """CTA pairs on 256 x 192 tiles (XMOD_PAIR_BN=192) for the o-projection (staged x
    rows) and the down projection's gated scatter (staged x and a rows): the same dot
    products in the same k order as the single-CTA tiles, so the stream agrees bit for
    bit, and the oracle within the bf16 tolerance."""
    w = CASES_192[case]
    dt = w.dtype
    lw = I.layer_weights(w, 4)
    bias = I.router_bias(w)
    x = I.residual_stream(w)
    if kind == 1:
        x, _ = U.enforce_routing_margin(x, dt, lw["w_r"], bias, w.K)
    y192 = _run(X, w, kind, x, lw, bias, pairs=True, pair_bn=192)
    y_single = _run(X, w, kind, x, lw, bias, pairs=False)
    assert torch.equal(y192.view(torch.int16), y_single.view(torch.int16))
    ref = O.layer_fwd(oracle_dims(w), kind, w.K, 0, oracle_layer(lw, dt), I.to_f64(x, dt),
                      bias=bias)
    got = from_dev(y192, dt).reshape(w.B, w.T, w.d)
    U.assert_close(got, ref["y"], dt, "y", stored_ref=got)
