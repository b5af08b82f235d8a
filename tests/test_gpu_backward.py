"""GPU parity of the layer backward (xmod_layer_bwd) against the oracle's layer_bwd,
through the C ABI: dx, every weight gradient, dJ/dvarsigma and the Eq. 9 loss, for
sparse layers under Eq. 7 and Eq. 6 (with and without the Eq. 9 term), dense layers, the
QK-norm / RoPE extras, the FullAttn / Routed-FFN halves and the Selected-Q / full-KV
control; and the stack backward.

Tolerances. fp32 (FFMA kernels throughout): relative 1e-5 as for the forward. bf16:
relative L2 <= 1e-2 (the bound of the bf16 forward); a gradient has no natural unit,
so the max-abs bound 2e-2 is taken relative to the gradient's largest reference entry.
The scalar dJ/dvarsigma, a sum of terms of both signs, is bounded by the same relative
figure times the L2 norm of its terms.
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


def _run(X, w: I.Workload, kind, gate, route_coef, seed, extras=None, path=None):
    """path: "as stored" -- the gradient GEMMs and the attention backward read their
    operands as stored, so the only transpose left is the rows' lse per head (at most two
    launches); "transposed" -- the weights and the activations are transposed for the
    gradient GEMMs (a weight launch and one per weight gradient)."""
    lw = I.layer_weights(w, 0)
    lw["varsigma"] = 0.9
    theta = 0.0
    if extras:   # QK-norm gains (non-trivial) and the rotary base
        ge = np.random.default_rng(seed + 1)
        for k in ("gq", "gk"):
            gains = (1 + 0.2 * ge.standard_normal(w.hd)).astype(np.float32)
            lw[k] = I.f32_to_bf16_bits(gains) if w.dtype == "bf16" else gains
        theta = extras
        lw["rope_theta"] = theta
    bias = I.router_bias(w)
    x = I.residual_stream(w)
    routed = kind in (X.LAYER_SPARSE, X.LAYER_ROUTED_FFN, X.LAYER_SPARSE_FULLKV)
    if routed:
        x, _ = U.enforce_routing_margin(x, w.dtype, lw["w_r"], bias, w.K)
    g = np.random.default_rng(seed)
    dyf = g.standard_normal((w.B, w.T, w.d)).astype(np.float32)
    dy = I.f32_to_bf16_bits(dyf) if w.dtype == "bf16" else dyf
    dm = xmod_dims(w)
    ws = torch.zeros(X.bwd_workspace_bytes(dm, w.K), dtype=torch.uint8, device="cuda")
    abi = X.layer_weights(dev_layer(lw, w.dtype), lw["varsigma"], theta)
    xd, dyd = to_dev(x, w.dtype), to_dev(dy, w.dtype)
    dx = torch.empty_like(xd)
    qw, kw = w.hq * w.hd, w.hkv * w.hd
    shapes = {"w_router": (w.d,), "rms1": (w.d,), "wq": (qw, w.d), "wk": (kw, w.d),
              "wv": (kw, w.d), "wo": (w.d, qw), "rms2": (w.d,), "w_gate": (w.F, w.d),
              "w_up": (w.F, w.d), "w_down": (w.d, w.F), "varsigma": (4,), "route_loss": (4,)}
    if extras:
        shapes["q_norm"] = shapes["k_norm"] = (w.hd,)
    gd = {k: torch.full(v, float("nan"), dtype=torch.float32, device="cuda")
          for k, v in shapes.items()}
    X.reset_status(ws)
    if path:
        X.profile_enable(True)
        X.profile_read()
    X.layer_bwd(dm, kind, w.K, gate, abi, xd, torch.from_numpy(bias).cuda()
                if bias is not None else None, dyd, route_coef, dx, X.layer_grads(gd), ws)
    assert X.sync_status(ws) == X.OK
    if path:
        n_tr = X.profile_read().get("bwd_transpose", (0, 0.0))[0]
        X.profile_enable(False)
        if path == "as stored":
            assert n_tr <= 2, f"{n_tr} transpose launches on the as-stored path"
        else:
            assert n_tr >= 5, f"only {n_tr} transpose launches on the transposed path"
    ref = O.layer_bwd(U_dims(w), kind, w.K, gate, oracle_layer(lw, w.dtype), I.to_f64(x, w.dtype),
                      I.to_f64(dy, w.dtype), bias=bias, route_coef=route_coef)
    _check(from_dev(dx, w.dtype), ref["dx"], w.dtype, "dx")
    for on, an in GRAD_NAMES.items():   # unused weights: zero on both sides
        _check(gd[an].cpu().numpy(), ref["grads"][on], w.dtype, f"d{on}")
    if extras:
        _check(gd["q_norm"].cpu().numpy(), ref["grads"]["gq"], w.dtype, "dq_norm")
        _check(gd["k_norm"].cpu().numpy(), ref["grads"]["gk"], w.dtype, "dk_norm")
    vs = float(gd["varsigma"][0])
    if routed and gate == X.GATE_XMOD:
        # dJ/dvarsigma = sum over the selected rows of r <dy, a + f> (Eq. 7): a sum whose
        # terms cancel, so its error is bounded on the scale of the terms, r dy (a + f) =
        # dy (y - x) / varsigma elementwise, as every other gradient is bounded on its own
        x64 = I.to_f64(x, w.dtype)
        fw = O.layer_fwd(U_dims(w), kind, w.K, gate, oracle_layer(lw, w.dtype), x64, bias=bias,
                         idx_force=ref["idx"])
        terms = I.to_f64(dy, w.dtype) * (fw["y"] - x64) / lw["varsigma"]
        tol = (U.FP32_REL if w.dtype == "fp32" else U.BF16_REL_L2) * float(np.linalg.norm(terms))
        assert np.isfinite(vs) and abs(vs - ref["varsigma"]) <= tol, \
            f"dvarsigma: {vs} vs {ref['varsigma']} (bound {tol:.2e})"
    else:
        assert vs == 0.0
    if routed:
        _check(np.array([float(gd["route_loss"][0])]), np.array([ref["route_loss"]]), w.dtype,
               "route loss")
    if routed and route_coef == 0.0:
        # a skipped token's gradient is the upstream gradient, bit for bit (full-KV: a
        # token that is also no selected query's key, i.e. after the last selected one)
        sel = np.zeros((w.B, w.T), bool)
        np.put_along_axis(sel, ref["idx"], True, 1)
        if kind == X.LAYER_SPARSE_FULLKV:
            sel |= np.arange(w.T)[None, :] <= ref["idx"].max(axis=1, keepdims=True)
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
    """bf16, head_dim 128 (tensor-core projections and gradients, the gradient GEMMs on
    operands as stored): A4K8-shaped heads at a reduced width, ragged row counts (n = 101:
    token rows past the count read as zero), both gates, the Eq. 9 term, a dense layer."""
    w = I.WORKLOADS["a4k8_bf16"].replace(B=2, T=T, K=K, d=256, hq=4, hkv=2, F=512, seed=31,
                                         weight_std=0.02 * np.sqrt(1536 / 256))
    _run(X, w, kind, gate, coef, seed=40 + T + K, path="as stored")


@pytest.mark.parametrize("T,K,kind", [(256, 4, 1), (303, 3, 1), (160, 1, 0)])
def test_layer_bwd_bf16_transposed_operands(X, T, K, kind):
    """bf16 whose model and FFN widths are not multiples of 64 (d = 288, F = 480): the
    gradient GEMMs cannot read their operands as stored (whole 64-column chunks) and get
    them transposed, on the K-major tensor-core GEMM; ragged row counts included."""
    w = I.WORKLOADS["a4k8_bf16"].replace(B=2, T=T, K=K, d=288, hq=2, hkv=1, F=480, seed=43,
                                         weight_std=0.02 * np.sqrt(1536 / 288))
    _run(X, w, kind, X.GATE_XMOD, 0.1 if kind else 0.0, seed=170 + T + K,
         path="transposed")


@pytest.mark.parametrize("dtype,kind,T", [("fp32", 1, 64), ("fp32", 0, 64), ("bf16", 1, 256),
                                          ("bf16", 0, 160)])
def test_layer_bwd_qk_norm_rope(X, dtype, kind, T):
    """With QK-norm gains and the rotary embedding (base 1e4) at the tokens' original
    positions: dx, every weight gradient and the two gains' gradients."""
    if dtype == "fp32":
        w = I.WORKLOADS["tiny_fp32"].replace(T=T)
    else:
        w = I.WORKLOADS["a4k8_bf16"].replace(B=2, T=T, K=4, d=256, hq=4, hkv=2, F=512, seed=33,
                                             weight_std=0.02 * np.sqrt(1536 / 256))
    _run(X, w, kind, X.GATE_XMOD, 0.1, seed=60 + T + kind, extras=1e4)


@pytest.mark.parametrize("dtype,kind,gate,coef", [("fp32", 2, 0, 0.0), ("fp32", 3, 0, 0.3),
                                                 ("fp32", 3, 1, 0.0), ("bf16", 2, 0, 0.0),
                                                 ("bf16", 3, 0, 0.1), ("bf16", 3, 1, 0.0)])
def test_layer_bwd_mechanism_controls(X, dtype, kind, gate, coef):
    """The FullAttn (ATTN) and Routed-FFN (ROUTED_FFN) halves of the block."""
    if dtype == "fp32":
        w = I.WORKLOADS["tiny_fp32"]
    else:
        w = I.WORKLOADS["a4k8_bf16"].replace(B=2, T=256, K=4, d=256, hq=4, hkv=2, F=512, seed=35,
                                             weight_std=0.02 * np.sqrt(1536 / 256))
    _run(X, w, kind, gate, coef, seed=80 + 5 * kind + gate)


@pytest.mark.parametrize("dtype,T,K,gate,coef,extras", [
    ("fp32", 64, 4, 0, 0.0, None), ("fp32", 64, 4, 1, 0.3, None), ("fp32", 64, 4, 0, 0.1, 1e4),
    ("bf16", 256, 4, 0, 0.1, None), ("bf16", 303, 3, 1, 0.0, None), ("bf16", 256, 8, 0, 0.0, 1e4)])
def test_layer_bwd_fullkv(X, dtype, T, K, gate, coef, extras):
    """The Selected-Q / full-KV control (SPARSE_FULLKV): the selected tokens' queries over
    every token's keys and values, so the gradient also reaches unselected rows; both
    gates, the Eq. 9 term, the QK-norm / RoPE extras, a ragged count (n = 101 of 303)."""
    if dtype == "fp32":
        w = I.WORKLOADS["tiny_fp32"].replace(T=T, K=K)
    else:
        w = I.WORKLOADS["a4k8_bf16"].replace(B=2, T=T, K=K, d=256, hq=4, hkv=2, F=512, seed=37,
                                             weight_std=0.02 * np.sqrt(1536 / 256))
    _run(X, w, X.LAYER_SPARSE_FULLKV, gate, coef, seed=120 + T + K + gate, extras=extras)


@pytest.mark.parametrize("kind,T,K", [(1, 256, 4), (1, 303, 3), (0, 160, 1), (4, 256, 4),
                                      (4, 303, 3)])
def test_layer_bwd_bf16_head_dim_64(X, kind, T, K):
    """bf16 at head_dim 64: the attention backward on the warp-level tensor-core MMA kernels
    (the tcgen05 pair takes head_dim 128), for sparse, dense and Selected-Q / full-KV
    layers, ragged counts included."""
    w = I.WORKLOADS["a4k8_bf16"].replace(B=2, T=T, K=K, d=256, hq=4, hkv=2, hd=64, F=512,
                                         seed=39, weight_std=0.02 * np.sqrt(1536 / 256))
    _run(X, w, kind, X.GATE_XMOD, 0.1 if kind else 0.0, seed=140 + T + K + kind)


def _grad_set(w, n_layers):
    qw, kw = w.hq * w.hd, w.hkv * w.hd
    shapes = {"w_router": (w.d,), "rms1": (w.d,), "wq": (qw, w.d), "wk": (kw, w.d),
              "wv": (kw, w.d), "wo": (w.d, qw), "rms2": (w.d,), "w_gate": (w.F, w.d),
              "w_up": (w.F, w.d), "w_down": (w.d, w.F), "varsigma": (4,), "route_loss": (4,)}
    return [{k: torch.full(v, float("nan"), dtype=torch.float32, device="cuda")
             for k, v in shapes.items()} for _ in range(n_layers)]


def _stack_case(X, w):
    from oracle import structure as S
    layers = I.all_layer_weights(w)
    kinds = S.schedule(w.N0, w.N1, w.A, w.K)
    bias = I.router_bias(w)
    x = I.residual_stream(w)
    x, _ = U.enforce_routing_margin(x, w.dtype, layers[kinds.index(S.SPARSE)]["w_r"], bias, w.K)
    g = np.random.default_rng(77)
    dyf = g.standard_normal((w.B, w.T, w.d)).astype(np.float32)
    dy = I.f32_to_bf16_bits(dyf) if w.dtype == "bf16" else dyf
    abi = [X.layer_weights(dev_layer(l, w.dtype), l["varsigma"]) for l in layers]
    return layers, kinds, bias, x, dy, abi


def test_stack_bwd_fp32_tiny_against_oracle(X):
    """xmod_stack_bwd on the tiny fp32 stack (Dense + 4 Sparse(4) + Dense) against the
    oracle's layer backward chained from the last layer to the first on the oracle's own
    forward layer inputs."""
    w = I.WORKLOADS["tiny_fp32"]
    layers, kinds, bias, x, dy, abi = _stack_case(X, w)
    coef = 0.3
    dm = xmod_dims(w)
    ws = torch.zeros(X.stack_bwd_workspace_bytes(dm, w.K), dtype=torch.uint8, device="cuda")
    ck = torch.empty((len(kinds), w.B, w.T, w.d), dtype=torch.float32, device="cuda")
    xd, dyd = to_dev(x, "fp32"), to_dev(dy, "fp32")
    dx = torch.empty_like(xd)
    gd = _grad_set(w, len(kinds))
    X.reset_status(ws)
    X.stack_bwd(dm, w.K, w.A, w.N0, w.N1, w.gate, abi, xd, torch.from_numpy(bias).cuda(), dyd,
                coef, dx, [X.layer_grads(g) for g in gd], ck, ws)
    assert X.sync_status(ws) == X.OK
    od = U_dims(w)
    ol = [oracle_layer(l, "fp32") for l in layers]
    xs = [I.to_f64(x, "fp32")]
    for l, kind in enumerate(kinds[:-1]):
        xs.append(O.layer_fwd(od, kind, w.K, w.gate, ol[l], xs[-1],
                              bias=bias if kind == O.SPARSE else None)["y"])
    g = I.to_f64(dy, "fp32")
    for l in range(len(kinds) - 1, -1, -1):
        kind = kinds[l]
        r = O.layer_bwd(od, kind, w.K, w.gate, ol[l], xs[l], g,
                        bias=bias if kind == O.SPARSE else None, route_coef=coef)
        for on, an in GRAD_NAMES.items():
            if kind == O.DENSE and on == "w_r":
                continue
            _check(gd[l][an].cpu().numpy(), r["grads"][on], "fp32", f"layer {l} d{on}")
        g = r["dx"]
    _check(from_dev(dx, "fp32"), g, "fp32", "stack dx")


def test_stack_bwd_bf16_equals_layer_chain(X):
    """bf16 (tensor-core path): xmod_stack_bwd equals, bit for bit, xmod_layer_fwd
    checkpoints followed by xmod_layer_bwd chained by hand."""
    w = I.WORKLOADS["a4k8_bf16"].replace(B=2, T=256, A=1, n_layers=9, d=256, hq=4, hkv=2,
                                         F=512, seed=5, weight_std=0.02 * np.sqrt(1536 / 256))
    layers, kinds, bias, x, dy, abi = _stack_case(X, w)
    coef = 1e-2
    dm = xmod_dims(w)
    bd = torch.from_numpy(bias).cuda()
    ws = torch.zeros(X.stack_bwd_workspace_bytes(dm, w.K), dtype=torch.uint8, device="cuda")
    ck = torch.empty((len(kinds), w.B, w.T, w.d), dtype=torch.bfloat16, device="cuda")
    xd, dyd = to_dev(x, "bf16"), to_dev(dy, "bf16")
    dx = torch.empty_like(xd)
    gd = _grad_set(w, len(kinds))
    X.reset_status(ws)
    X.stack_bwd(dm, w.K, w.A, w.N0, w.N1, w.gate, abi, xd, bd, dyd, coef, dx,
                [X.layer_grads(g) for g in gd], ck, ws)
    assert X.sync_status(ws) == X.OK
    # by hand
    wsf = torch.zeros(X.workspace_bytes(dm, w.K), dtype=torch.uint8, device="cuda")
    wsb = torch.zeros(X.bwd_workspace_bytes(dm, w.K), dtype=torch.uint8, device="cuda")
    xs = [xd.clone()]
    for l, kind in enumerate(kinds[:-1]):
        nxt = xs[-1].clone()
        X.layer_fwd(dm, kind, w.K, w.gate, abi[l], nxt, bd if kind == X.LAYER_SPARSE else None,
                    None, None, wsf)
        xs.append(nxt)
    for l in range(len(kinds)):
        assert torch.equal(ck[l].view(torch.int16), xs[l].view(torch.int16)), f"checkpoint {l}"
    g = dyd
    hand = _grad_set(w, len(kinds))
    for l in range(len(kinds) - 1, -1, -1):
        out = torch.empty_like(xd)
        X.layer_bwd(dm, kinds[l], w.K, w.gate, abi[l], xs[l],
                    bd if kinds[l] == X.LAYER_SPARSE else None, g, coef, out,
                    X.layer_grads(hand[l]), wsb)
        g = out
    assert X.sync_status(wsb) == X.OK
    assert torch.equal(dx.view(torch.int16), g.view(torch.int16))
    for l in range(len(kinds)):
        for k in ("w_router", "rms1", "wq", "wk", "wv", "wo", "rms2", "w_gate", "w_up", "w_down",
                  "varsigma"):
            if kinds[l] == X.LAYER_DENSE and k == "w_router":
                continue
            a, b = gd[l][k], hand[l][k]
            if k == "varsigma":
                a, b = a[:1], b[:1]
            assert torch.equal(a, b), f"layer {l} {k}"


def _bwd_once(X, w, kind, lw, x, dy, bias, pairs):
    import os
    dm = xmod_dims(w)
    ws = torch.zeros(X.bwd_workspace_bytes(dm, w.K), dtype=torch.uint8, device="cuda")
    abi = X.layer_weights(dev_layer(lw, w.dtype), lw["varsigma"], 0.0)
    xd, dyd = to_dev(x, w.dtype), to_dev(dy, w.dtype)
    dx = torch.empty_like(xd)
    gd = _grad_set(w, 1)[0]
    old = {k: os.environ.get(k) for k in ("XMOD_PAIR_MIN_WAVES", "XMOD_STREAM_K")}
    os.environ["XMOD_PAIR_MIN_WAVES"] = "0" if pairs else "999999"
    os.environ["XMOD_STREAM_K"] = "0"
    try:
        X.reset_status(ws)
        X.layer_bwd(dm, kind, w.K, X.GATE_XMOD, abi, xd,
                    torch.from_numpy(bias).cuda() if bias is not None else None, dyd, 0.1, dx,
                    X.layer_grads(gd), ws)
        assert X.sync_status(ws) == X.OK
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return dx, gd


@pytest.mark.parametrize("kind", [0, 1, 4])
def test_layer_bwd_on_cta_pairs_equals_single_ctas(X, kind):
    """Every GEMM of the backward on CTA pairs (XMOD_PAIR_MIN_WAVES=0) against the same
    call on single CTAs: the pair and single kernels form each output element as the same
    dot product in the same k order, so dx and every gradient agree bit for bit -- this
    covers the pair kernel's q|k|v epilogue writing v both transposed and by rows, and its
    fp32 store splitting the stacked weight gradients by rows. Dense, sparse and full-KV."""
    w = I.WORKLOADS["a4k8_bf16"].replace(B=2, T=512, K=4, d=256, hq=4, hkv=2, F=384, seed=43,
                                         weight_std=0.049)
    lw = I.layer_weights(w, 0)
    lw["varsigma"] = 0.9
    bias = I.router_bias(w)
    x = I.residual_stream(w)
    if kind:
        x, _ = U.enforce_routing_margin(x, w.dtype, lw["w_r"], bias, w.K)
    dyf = np.random.default_rng(44).standard_normal((w.B, w.T, w.d)).astype(np.float32)
    dy = I.f32_to_bf16_bits(dyf)
    dx1, g1 = _bwd_once(X, w, kind, lw, x, dy, bias, pairs=True)
    dx0, g0 = _bwd_once(X, w, kind, lw, x, dy, bias, pairs=False)
    assert torch.equal(dx1.view(torch.int16), dx0.view(torch.int16))
    for k in ("rms1", "wq", "wk", "wv", "wo", "rms2", "w_gate", "w_up", "w_down", "varsigma"):
        assert torch.equal(g1[k].view(torch.int32), g0[k].view(torch.int32)), k
