"""GPU parity of the routing kernels (router, top-(T/K), gather, gated scatter)
against the CPU oracle, through the C ABI."""
import numpy as np
import pytest

import oracle as O
from sparse_depth_token_gb300 import inputs as I
from tests import _util as U
from tests._gpu import (dev_layer, from_dev, need_gpu, to_dev, torch, workspace, xmod_dims)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def X():
    need_gpu()
    from sparse_depth_token_gb300 import xmod
    xmod.load()
    return xmod


def _logits(kind, B, T, seed):
    g = np.random.default_rng(seed)
    s = g.standard_normal((B, T)).astype(np.float32)
    if kind == "ties":
        s = (np.round(s * 4) / 4).astype(np.float32)
    elif kind == "equal":
        s = np.full((B, T), 0.5, np.float32)
    elif kind == "zeros":
        s = np.where(g.random((B, T)) < 0.5, np.float32(-0.0), np.float32(0.0))
        s[:, ::7] = -1.0
    elif kind == "wide":
        s = (s * np.float32(1e30)).astype(np.float32)
    return s


@pytest.mark.parametrize("B,T,K", [(3, 64, 4), (2, 1000, 3), (4, 4096, 8), (2, 8192, 2),
                                   (2, 16384, 16), (1, 7, 7), (2, 1025, 1)])
@pytest.mark.parametrize("kind", ["normal", "ties", "equal", "zeros", "wide"])
def test_topk_on_given_logits_bit_exact(X, B, T, K, kind):
    s = _logits(kind, B, T, B * T + K)
    n = T // K
    dm = X.dims(B, T, 8, 1, 1, 8, 8, X.FP32)
    ws = workspace(dm, K)
    s_d = torch.from_numpy(s).cuda()
    idx = torch.empty((B, n), dtype=torch.int32, device="cuda")
    r_sel = torch.empty((B, n), dtype=torch.float32, device="cuda")
    X.reset_status(ws)
    X.topk(dm, K, s_d, idx, r_sel, ws)
    assert X.sync_status(ws) == X.OK
    ref = O.topk(s.astype(np.float64), n)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref)
    r_ref = 1.0 / (1.0 + np.exp(-np.take_along_axis(s.astype(np.float64), ref, 1)))
    np.testing.assert_allclose(r_sel.cpu().numpy(), r_ref, rtol=2e-6, atol=1e-30)


def test_topk_nonfinite_logit_sets_status(X):
    B, T, K = 2, 256, 4
    s = _logits("normal", B, T, 5)
    s[1, 17] = np.nan
    dm = X.dims(B, T, 8, 1, 1, 8, 8, X.FP32)
    ws = workspace(dm, K)
    idx = torch.empty((B, T // K), dtype=torch.int32, device="cuda")
    X.reset_status(ws)
    X.topk(dm, K, torch.from_numpy(s).cuda(), idx, None, ws)
    assert X.sync_status(ws) == X.ERR_DEVICE_CHECK
    X.reset_status(ws)
    assert X.sync_status(ws) == X.OK
    # the selection is still a permutation-free ascending list of n positions
    got = idx.cpu().numpy()
    assert np.all(np.diff(got, axis=1) > 0)


def _routing_case(w: I.Workload, K):
    x = I.residual_stream(w)
    lw = I.layer_weights(w, 0)
    bias = I.router_bias(w)
    x, touched = U.enforce_routing_margin(x, w.dtype, lw["w_r"], bias, K)
    return x, lw, bias


@pytest.mark.parametrize("dtype,K,with_bias", [("bf16", 8, False), ("bf16", 2, True),
                                               ("fp32", 4, True), ("bf16", 16, False)])
def test_router_topk_bit_exact_small(X, dtype, K, with_bias):
    w = I.WORKLOADS["routing_bf16"].replace(B=4, T=2000, d=512, dtype=dtype, seed=11,
                                            bias_std=0.1 if with_bias else 0.0)
    x, lw, bias = _routing_case(w, K)
    n = w.T // K
    dm = xmod_dims(w)
    ws = workspace(dm, K)
    xd = to_dev(x, dtype)
    wr = to_dev(lw["w_r"], dtype)
    bd = torch.from_numpy(bias).cuda() if bias is not None else None
    logits = torch.empty((w.B, w.T), dtype=torch.float32, device="cuda")
    r = torch.empty_like(logits)
    idx = torch.empty((w.B, n), dtype=torch.int32, device="cuda")
    r_sel = torch.empty((w.B, n), dtype=torch.float32, device="cuda")
    X.reset_status(ws)
    X.router_topk(dm, K, xd, wr, bd, logits, r, idx, r_sel, ws)
    assert X.sync_status(ws) == X.OK
    s_ref, r_ref = O.router(I.to_f64(x, dtype), I.to_f64(lw["w_r"], dtype), bias)
    np.testing.assert_allclose(logits.cpu().numpy(), s_ref, rtol=1e-5, atol=2e-6)
    np.testing.assert_allclose(r.cpu().numpy(), r_ref, rtol=1e-5, atol=1e-6)
    assert np.all(U.kth_gap(s_ref, n) >= U.ROUTING_MARGIN)
    idx_ref = O.topk(s_ref, n)
    np.testing.assert_array_equal(idx.cpu().numpy(), idx_ref)
    np.testing.assert_allclose(r_sel.cpu().numpy(), np.take_along_axis(r_ref, idx_ref, 1),
                               rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_gather_bit_exact(X, dtype):
    B, T, d, K = 3, 300, 136, 3
    g = np.random.default_rng(4)
    xf = g.standard_normal((B, T, d)).astype(np.float32)
    x = I.f32_to_bf16_bits(xf) if dtype == "bf16" else xf
    n = T // K
    idx = np.sort(np.stack([g.choice(T, n, replace=False) for _ in range(B)]), 1).astype(np.int32)
    dm = X.dims(B, T, d, 1, 1, 8, 8, X.BF16 if dtype == "bf16" else X.FP32)
    xs = torch.empty((B * n, d), dtype=torch.bfloat16 if dtype == "bf16" else torch.float32,
                     device="cuda")
    X.gather(dm, K, to_dev(x, dtype), torch.from_numpy(idx).cuda(), xs)
    torch.cuda.synchronize()
    ref = np.concatenate([I.to_f64(x[b, idx[b]], dtype) for b in range(B)])
    np.testing.assert_array_equal(from_dev(xs, dtype), ref)


@pytest.mark.parametrize("dtype,gate,fused_af", [("bf16", 0, False), ("bf16", 1, False),
                                                 ("bf16", 0, True), ("fp32", 0, False),
                                                 ("fp32", 1, False)])
def test_gated_scatter(X, dtype, gate, fused_af):
    B, T, d, K = 2, 96, 64, 4
    n = T // K
    g = np.random.default_rng(7 + gate)
    conv = (lambda a: I.f32_to_bf16_bits(a)) if dtype == "bf16" else (lambda a: a)
    x = conv(g.standard_normal((B, T, d)).astype(np.float32))
    a = conv(g.standard_normal((B * n, d)).astype(np.float32))
    f = conv(g.standard_normal((B * n, d)).astype(np.float32))
    r = g.random(B * n).astype(np.float32)
    idx = np.sort(np.stack([g.choice(T, n, replace=False) for _ in range(B)]), 1).astype(np.int32)
    vs = 1.25
    dm = X.dims(B, T, d, 1, 1, 8, 8, X.BF16 if dtype == "bf16" else X.FP32)
    xd = to_dev(x, dtype)
    af = conv((I.to_f64(a, dtype) + I.to_f64(f, dtype)).astype(np.float32))
    X.gated_scatter(dm, K, xd, torch.from_numpy(idx).cuda(), torch.from_numpy(r).cuda(),
                    to_dev(af if fused_af else a, dtype), None if fused_af else to_dev(f, dtype),
                    vs, gate)
    torch.cuda.synchronize()
    rows = (np.arange(B)[:, None] * T + idx).reshape(-1)
    a64, f64 = I.to_f64(a, dtype), I.to_f64(f, dtype)
    if fused_af:
        ref = O.gated_scatter(I.to_f64(x, dtype).reshape(-1, d), rows, I.to_f64(af, dtype), None,
                              r.astype(np.float64), vs, gate)
    else:
        ref = O.gated_scatter(I.to_f64(x, dtype).reshape(-1, d), rows, a64, f64,
                              r.astype(np.float64), vs, gate)
    got = from_dev(xd, dtype).reshape(-1, d)
    unsel = np.setdiff1d(np.arange(B * T), rows)
    np.testing.assert_array_equal(got[unsel], I.to_f64(x, dtype).reshape(-1, d)[unsel])
    U.assert_close(got[rows], ref[rows], dtype, "scatter")


@pytest.mark.slow
@pytest.mark.parametrize("K", [8])
def test_router_topk_full_routing_bench(X, K):
    """The routing microbench at full size (B=64, T=8192, d=4096, bf16), margin-fixed."""
    w = I.WORKLOADS["routing_bf16"]
    x, lw, bias = _routing_case(w, K)
    n = w.T // K
    dm = xmod_dims(w)
    ws = workspace(dm, K)
    xd = to_dev(x, "bf16")
    del x
    logits = torch.empty((w.B, w.T), dtype=torch.float32, device="cuda")
    idx = torch.empty((w.B, n), dtype=torch.int32, device="cuda")
    r_sel = torch.empty((w.B, n), dtype=torch.float32, device="cuda")
    X.reset_status(ws)
    X.router_topk(dm, K, xd, to_dev(lw["w_r"], "bf16"), None, logits, None, idx, r_sel, ws)
    assert X.sync_status(ws) == X.OK
    x64 = from_dev(xd, "bf16").reshape(w.B, w.T, w.d)
    s_ref, r_ref = O.router(x64, I.to_f64(lw["w_r"], "bf16"))
    np.testing.assert_allclose(logits.cpu().numpy(), s_ref, rtol=1e-5, atol=5e-6)
    np.testing.assert_array_equal(idx.cpu().numpy(), O.topk(s_ref, n))
