"""GPU parity of the Eq. 3 stack against the CPU oracle, through the C ABI.

End to end on the tiny fp32 stack; layer by layer (teacher-forced) on bf16
stacks, including the A4K8 block at its full size in the launch configuration
the benchmark times, where the oracle computes sampled rows one by one."""
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


def _setup(X, w: I.Workload, n_layers=None):
    layers = I.all_layer_weights(w, n_layers)
    kinds = S.schedule(w.N0, w.N1, w.A, w.K)
    assert len(kinds) == len(layers)
    bias = I.router_bias(w)
    x = I.residual_stream(w)
    first_sparse = kinds.index(S.SPARSE)
    x, _ = U.enforce_routing_margin(x, w.dtype, layers[first_sparse]["w_r"], bias, w.K)
    dev = [dev_layer(l, w.dtype) for l in layers]
    abi = [X.layer_weights(d, l["varsigma"]) for d, l in zip(dev, layers)]
    return layers, kinds, bias, x, dev, abi


def test_tiny_fp32_stack_end_to_end(X):
    w = I.WORKLOADS["tiny_fp32"]
    layers, kinds, bias, x, dev, abi = _setup(X, w)
    dm = xmod_dims(w)
    ws = workspace(dm, w.K)
    xd = to_dev(x, "fp32")
    bd = torch.from_numpy(bias).cuda()
    X.reset_status(ws)
    X.stack_fwd(dm, w.K, w.A, w.N0, w.N1, w.gate, abi, xd, bd, ws)
    assert X.sync_status(ws) == X.OK
    ref = O.stack_fwd(oracle_dims(w), w.K, w.gate, kinds, [oracle_layer(l, "fp32") for l in layers],
                      I.to_f64(x, "fp32"), bias=bias)
    U.assert_close(from_dev(xd, "fp32").reshape(ref.shape), ref, "fp32", "stack")


def _teacher_forced(X, w, layers, kinds, bias, x, abi, check_layers, row_mask=None):
    """Run the stack one layer at a time on the GPU; at the listed layers compare with
    the oracle run on the GPU layer's own input. Returns the final GPU stream."""
    dm = xmod_dims(w)
    ws = workspace(dm, w.K)
    od = oracle_dims(w)
    xd = to_dev(x, w.dtype)
    bd = torch.from_numpy(bias).cuda() if bias is not None else None
    n = w.T // w.K
    idx = torch.empty((w.B, n), dtype=torch.int32, device="cuda")
    r_sel = torch.empty((w.B, n), dtype=torch.float32, device="cuda")
    X.reset_status(ws)
    for l, kind in enumerate(kinds):
        x_in = from_dev(xd, w.dtype).reshape(w.B, w.T, w.d) if l in check_layers else None
        X.layer_fwd(dm, kind, w.K, w.gate, abi[l], xd, bd, idx if kind else None,
                    r_sel if kind else None, ws)
        if l not in check_layers:
            continue
        assert X.sync_status(ws) == X.OK
        L = oracle_layer(layers[l], w.dtype)
        got = from_dev(xd, w.dtype).reshape(w.B, w.T, w.d)
        force = None
        if kind == S.SPARSE:
            s, _ = O.router(x_in, I.to_f64(layers[l]["w_r"], w.dtype), bias)
            gidx = idx.cpu().numpy()
            differ = U.check_selection(gidx, s, n)
            if l == kinds.index(S.SPARSE) == 0:
                # the margin was enforced on the stack's input, which is this layer's input
                assert differ == 0, "first sparse layer has margin-fixed inputs: must be bit-exact"
            force = gidx
        ref = O.layer_fwd(od, kind, w.K, w.gate, L, x_in, bias=bias, idx_force=force,
                          row_mask=row_mask)
        m = np.ones((w.B, w.T), bool) if row_mask is None else row_mask.astype(bool)
        if kind == S.SPARSE:
            sel = np.zeros((w.B, w.T), bool)
            np.put_along_axis(sel, force, True, 1)
            np.testing.assert_array_equal(got[~sel], x_in[~sel])
            m = m & sel
        U.assert_close(got[m], ref["y"][m], w.dtype, f"layer {l} y", stored_ref=got[m])
        U.assert_close(got[m] - x_in[m], ref["y"][m] - x_in[m], w.dtype, f"layer {l} update",
                       stored_ref=got[m])
    assert X.sync_status(ws) == X.OK
    return xd, dm, ws


def test_tiny_fp32_teacher_forced(X):
    w = I.WORKLOADS["tiny_fp32"]
    layers, kinds, bias, x, dev, abi = _setup(X, w)
    _teacher_forced(X, w, layers, kinds, bias, x, abi, set(range(len(kinds))))


def _reduced(name):
    """The bf16 workloads at their widths and heads, shortened: B=2, T=512, one block."""
    base = I.WORKLOADS[name]
    if name == "a3k16_bf16":
        return base.replace(B=2, T=512, N0=1, N1=1, n_layers=1 + 49)
    if name == "mod_bf16":
        return base.replace(B=2, T=512, N1=2, n_layers=4)
    return base.replace(B=2, T=512, A=1, n_layers=9)


@pytest.mark.parametrize("name", ["a4k8_bf16", "mod_bf16", "a3k16_bf16"])
def test_bf16_stack_reduced_teacher_forced(X, name):
    """The bf16 workloads at their widths and heads, shortened: B=2, T=512, one block."""
    w = _reduced(name)
    layers, kinds, bias, x, dev, abi = _setup(X, w)
    xd, dm, ws = _teacher_forced(X, w, layers, kinds, bias, x, abi, set(range(len(kinds))))
    # the stack entry point reproduces the layer-by-layer result bit for bit
    xs = to_dev(x, w.dtype)
    X.stack_fwd(dm, w.K, w.A, w.N0, w.N1, w.gate, abi, xs,
                torch.from_numpy(bias).cuda() if bias is not None else None, ws)
    assert X.sync_status(ws) == X.OK
    assert torch.equal(xs.view(torch.int16), xd.view(torch.int16))


@pytest.mark.parametrize("name", ["a4k8_bf16", "a3k16_bf16"])
def test_stack_captured_in_a_cuda_graph(X, name):
    """xmod_stack_fwd is capture-safe: the call recorded once into a CUDA graph on a side
    stream (its launches, with their programmatic-launch edges, become graph nodes) and
    replayed twice over a fresh copy of the input gives the eager call's stream bit for
    bit; the status word stays clear."""
    w = _reduced(name)
    layers, kinds, bias, x, dev, abi = _setup(X, w)
    dm = xmod_dims(w)
    ws = workspace(dm, w.K)
    bd = torch.from_numpy(bias).cuda() if bias is not None else None
    x0 = to_dev(x, w.dtype)
    eager = x0.clone()
    X.reset_status(ws)
    X.stack_fwd(dm, w.K, w.A, w.N0, w.N1, w.gate, abi, eager, bd, ws)
    assert X.sync_status(ws) == X.OK
    xs = torch.empty_like(x0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):   # warm the stream (first-use work stays out of the capture)
        xs.copy_(x0)
        X.stack_fwd(dm, w.K, w.A, w.N0, w.N1, w.gate, abi, xs, bd, ws, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        xs.copy_(x0)
        X.stack_fwd(dm, w.K, w.A, w.N0, w.N1, w.gate, abi, xs, bd, ws, stream=s)
    for _ in range(2):
        xs.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(xs.view(torch.int16), eager.view(torch.int16))
    assert X.sync_status(ws) == X.OK


@pytest.mark.parametrize("name", ["a4k8_bf16", "mod_bf16", "a3k16_bf16"])
def test_bf16_stack_reduced_end_to_end(X, name):
    """End to end, with no teacher forcing of the stream: xmod_stack_fwd on the shortened
    bf16 stacks against the oracle's own storage-mirroring stack (its residual stream
    rounded to bf16 after every layer). Only routing decisions are shared. At every
    sparse layer the GPU's selection must be a valid top-(T/K) of the oracle's logits on
    the GPU's own input to that layer (up to the 1e-4 near-tie band, the teacher-forced
    routing criterion); the oracle layer then takes that selection, and the layers where
    the oracle's own stream would have chosen other tokens are counted and reported --
    the two streams differ by rounding, so near the k-th rank a layer may legitimately
    pick differently, which moves the tokens it updates.
    Bar: relative L2 <= 1e-2 over the whole final stream; max-abs reported; the first
    sparse layer routes on the margin-fixed input and must match bit for bit."""
    w = _reduced(name)
    layers, kinds, bias, x, dev, abi = _setup(X, w)
    dm = xmod_dims(w)
    ws = workspace(dm, w.K)
    bd = torch.from_numpy(bias).cuda() if bias is not None else None
    xs = to_dev(x, w.dtype)
    X.reset_status(ws)
    X.stack_fwd(dm, w.K, w.A, w.N0, w.N1, w.gate, abi, xs, bd, ws)
    assert X.sync_status(ws) == X.OK
    got = from_dev(xs, w.dtype).reshape(w.B, w.T, w.d)
    # the GPU's per-layer inputs and selections (the layer sequence equals the stack bit
    # for bit)
    n = w.T // w.K
    xd = to_dev(x, w.dtype)
    idx = torch.empty((w.B, n), dtype=torch.int32, device="cuda")
    gpu_in, gpu_idx = {}, {}
    for l, kind in enumerate(kinds):
        if kind:
            gpu_in[l] = from_dev(xd, w.dtype).reshape(w.B, w.T, w.d)
        X.layer_fwd(dm, kind, w.K, w.gate, abi[l], xd, bd, idx if kind else None, None, ws)
        if kind:
            gpu_idx[l] = idx.cpu().numpy()
    assert X.sync_status(ws) == X.OK
    assert torch.equal(xd.view(torch.int16), xs.view(torch.int16))
    # the oracle's own stream, layer by layer, bf16-mirrored, with the GPU's selections
    od = oracle_dims(w)
    xo = I.to_f64(x, w.dtype)
    differ = []
    first_sparse = kinds.index(S.SPARSE)
    for l, kind in enumerate(kinds):
        L = oracle_layer(layers[l], w.dtype)
        force = None
        if kind == S.SPARSE:
            wr = I.to_f64(layers[l]["w_r"], w.dtype)
            force = gpu_idx[l]
            s_gpu_in, _ = O.router(gpu_in[l], wr, bias)
            nd = U.check_selection(force, s_gpu_in, n)   # teacher-forced routing criterion
            if l == first_sparse == 0:
                assert nd == 0, "the first layer routes on the margin-fixed input: bit-exact"
            own = O.topk(O.router(xo, wr, bias)[0], n)
            if not np.array_equal(own, force):
                differ.append(l)
        xo = O.round_bf16_array(O.layer_fwd(od, kind, w.K, w.gate, L, xo, bias=bias,
                                            idx_force=force)["y"])
    rel = U.rel_l2(got, xo)
    mx = float(np.max(np.abs(got - xo)))
    print(f"{name} reduced stack end to end: rel-L2 {rel:.3e}, max-abs {mx:.3e}; at "
          f"{len(differ)} of {len(gpu_idx)} sparse layers the oracle's own stream would have "
          f"selected differently {differ}")
    assert rel <= U.BF16_REL_L2, f"{name}: end-to-end rel-L2 {rel:.3e}"


@pytest.mark.slow
def test_a4k8_full_size_sampled(X):
    """A4K8 block (32 Sparse(8) + Dense, d=1536, B=8, T=4096) at full size: sampled rows of
    the first, a middle and the last sparse layer and of the dense anchor."""
    w = I.WORKLOADS["a4k8_bf16"]
    layers, kinds, bias, x, dev, abi = _setup(X, w)
    mask = np.zeros((w.B, w.T), np.int32)
    g = np.random.default_rng(0)
    for b in (0, w.B - 1):
        mask[b, g.choice(w.T, 48, replace=False)] = 1
        mask[b, :4] = 1
        mask[b, -4:] = 1
    xd, dm, ws = _teacher_forced(X, w, layers, kinds, bias, x, abi, {0, 16, 31, 32}, row_mask=mask)
    xs = to_dev(x, w.dtype)
    X.stack_fwd(dm, w.K, w.A, w.N0, w.N1, w.gate, abi, xs, torch.from_numpy(bias).cuda(), ws)
    assert X.sync_status(ws) == X.OK
    assert torch.equal(xs.view(torch.int16), xd.view(torch.int16))
