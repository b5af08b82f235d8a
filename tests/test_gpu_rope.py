"""GPU: QK-norm and rotary position embedding at the tokens' original positions (the
Qwen3-style attention of the backbones the X-MoD notes train; NEXT row "RoPE at
original positions, QK-norm") against the oracle, in every layer kind that attends:
dense, sparse (compact rows rotated at their original positions), the FullAttn half,
Selected-Q / full-KV (queries at selected positions, keys at every position), and the
threshold rule (variable rows per sequence)."""
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
THETA = 1e4


@pytest.fixture(scope="module")
def X():
    need_gpu()
    from sparse_depth_token_gb300 import xmod
    xmod.load()
    return xmod


CASES = {
    "tiny_fp32": I.WORKLOADS["tiny_fp32"],
    "bf16_small": I.WORKLOADS["a4k8_bf16"].replace(B=2, T=512, d=256, hq=4, hkv=2, F=384,
                                                   seed=101, weight_std=0.049),
}


def _layer(w, seed):
    lw = I.layer_weights(w, seed)
    g = np.random.default_rng(seed)
    dt = np.float32
    lw["gq"] = (1 + 0.1 * g.standard_normal(w.hd)).astype(dt)
    lw["gk"] = (1 + 0.1 * g.standard_normal(w.hd)).astype(dt)
    if w.dtype == "bf16":   # the gains are stored in bf16 like every weight
        lw["gq"] = I.f32_to_bf16_bits(lw["gq"])
        lw["gk"] = I.f32_to_bf16_bits(lw["gk"])
    lw["rope_theta"] = THETA
    return lw


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("kind", [S.DENSE, S.SPARSE, S.ATTN, FULLKV])
def test_rope_qknorm_layer_against_oracle(X, case, kind):
    w = CASES[case]
    dt = w.dtype
    lw = _layer(w, 7)
    bias = I.router_bias(w)
    x = I.residual_stream(w)
    if kind in (S.SPARSE, FULLKV):
        x, _ = U.enforce_routing_margin(x, dt, lw["w_r"], bias, w.K)
    dm = xmod_dims(w)
    ws = workspace(dm, w.K)
    xd = to_dev(x, dt)
    X.reset_status(ws)
    X.layer_fwd(dm, kind, w.K, 0, X.layer_weights(dev_layer(lw, dt), lw["varsigma"], THETA), xd,
                torch.from_numpy(bias).cuda() if bias is not None else None, None, None, ws)
    assert X.sync_status(ws) == X.OK
    ref = O.layer_fwd(oracle_dims(w), kind, w.K, 0, oracle_layer(lw, dt), I.to_f64(x, dt),
                      bias=bias)
    got = from_dev(xd, dt).reshape(w.B, w.T, w.d)
    U.assert_close(got, ref["y"], dt, "y", stored_ref=got)
    x64 = I.to_f64(x, dt)
    if kind in (S.SPARSE, FULLKV):
        sel = np.zeros((w.B, w.T), bool)
        np.put_along_axis(sel, ref["idx"], True, 1)
        np.testing.assert_array_equal(got[~sel], x64[~sel])


def test_rope_qknorm_threshold_layer(X):
    w = CASES["bf16_small"]
    lw = _layer(w, 8)
    x = I.residual_stream(w)
    bias = I.router_bias(w).astype(np.float64) + np.array([-0.7, 0.4])[:, None]
    s, _ = O.router(I.to_f64(x, "bf16"), I.to_f64(lw["w_r"], "bf16"), bias=bias)
    near = np.abs(s) < 1e-3
    bias[near] += np.where(s[near] >= 0, 2e-3, -2e-3)
    bias = bias.astype(np.float32)
    dm = xmod_dims(w)
    ws = workspace(dm, w.K)
    xd = to_dev(x, "bf16")
    X.reset_status(ws)
    X.layer_fwd_threshold(dm, 0, X.layer_weights(dev_layer(lw, "bf16"), lw["varsigma"], THETA), xd,
                          torch.from_numpy(bias).cuda(), ws)
    assert X.sync_status(ws) == X.OK
    y, s, mask = O.layer_threshold(oracle_dims(w), 0, oracle_layer(lw, "bf16"),
                                   I.to_f64(x, "bf16"), bias=bias.astype(np.float64))
    got = from_dev(xd, "bf16").reshape(w.B, w.T, w.d)
    U.assert_close(got, y, "bf16", "y", stored_ref=got)
