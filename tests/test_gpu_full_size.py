"""GPU parity at the workloads' full sizes, in the launch configurations the benchmark
times, where the oracle computes sampled outputs one by one:

- the routing-only microbench (B=64, T=8192, d=4096, K in {2, 8, 16}): router logits,
  top-(T/K) indices (bit-exact), gates, the gathered rows (bit-exact) and the Eq. 7
  scatter of a given block output, on sampled sequences;
- the original MoD stack (([Sparse(8)] + [Dense]) x 4, Eq. 6, d=2048, B=4, T=8192) and
  the X-MoD A3K16 stack (N0=2, N1=2, 48 Sparse(16) layers per block, 100 layers, d=2048,
  B=4, T=16384), teacher-forced at sampled layers on sampled rows, and the stack entry
  point equal to the layer-by-layer composition bit for bit.
"""
import numpy as np
import pytest

import oracle as O
from sparse_depth_token_gb300 import inputs as I
from tests import _util as U
from tests._gpu import from_dev, need_gpu, to_dev, torch, workspace
from tests.test_gpu_stack import _setup, _teacher_forced

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def X():
    need_gpu()
    from sparse_depth_token_gb300 import xmod
    xmod.load()
    return xmod


def _row_mask(w, seqs, per_seq=48, seed=0):
    mask = np.zeros((w.B, w.T), np.int32)
    g = np.random.default_rng(seed)
    for b in seqs:
        mask[b, g.choice(w.T, per_seq, replace=False)] = 1
        mask[b, :4] = 1
        mask[b, -4:] = 1
    return mask


@pytest.fixture(scope="module")
def routing_stream():
    w = I.WORKLOADS["routing_bf16"]
    return w, I.residual_stream(w)


@pytest.mark.parametrize("K", [2, 8, 16])
def test_routing_microbench_full_size_sampled(X, routing_stream, K):
    """router_topk, gather and the Eq. 7 scatter of a given a+f at B=64, T=8192, d=4096,
    exactly as the benchmark calls them; the oracle checks four whole sequences."""
    w, x_all = routing_stream
    n = w.T // K
    M = w.B * n
    seqs = [0, 21, 42, w.B - 1]
    w_r = I.layer_weights(w, 0)["w_r"]
    x = np.array(x_all, copy=True)
    x[seqs], _ = U.enforce_routing_margin(x[seqs], "bf16", w_r, None, K)
    af = I.given_block_output(w, M)
    dm = X.dims(w.B, w.T, w.d, 1, 1, 8, 8, X.BF16, w.eps)
    ws = workspace(dm, K)
    xd = to_dev(x, "bf16")
    logits = torch.empty((w.B, w.T), dtype=torch.float32, device="cuda")
    idx = torch.empty((w.B, n), dtype=torch.int32, device="cuda")
    r_sel = torch.empty((w.B, n), dtype=torch.float32, device="cuda")
    xs = torch.empty((M, w.d), dtype=torch.bfloat16, device="cuda")
    X.reset_status(ws)
    X.router_topk(dm, K, xd, to_dev(w_r, "bf16"), None, logits, None, idx, r_sel, ws)
    X.gather(dm, K, xd, idx, xs)
    X.gated_scatter(dm, K, xd, idx, r_sel, to_dev(af, "bf16"), None, 1.0, X.GATE_XMOD)
    assert X.sync_status(ws) == X.OK
    w64 = I.to_f64(w_r, "bf16")
    for b in seqs:
        xb = I.to_f64(x[b], "bf16")
        s_ref, r_ref = O.router(xb, w64)
        np.testing.assert_allclose(logits[b].cpu().numpy(), s_ref, rtol=1e-5, atol=5e-6)
        assert U.kth_gap(s_ref[None], n)[0] >= U.ROUTING_MARGIN
        idx_ref = O.topk(s_ref[None], n)[0]
        gi = idx[b].cpu().numpy()
        np.testing.assert_array_equal(gi, idx_ref)
        np.testing.assert_allclose(r_sel[b].cpu().numpy(), r_ref[idx_ref], rtol=1e-5, atol=1e-6)
        # the gather: row j of sequence b is x[b, idx[j]], bit for bit
        np.testing.assert_array_equal(from_dev(xs[b * n:(b + 1) * n], "bf16"), xb[idx_ref])
        # the scatter: Eq. 7 on the selected rows, every other row untouched
        got = from_dev(xd[b], "bf16")
        af_b = I.to_f64(af[b * n:(b + 1) * n], "bf16")
        ref = O.gated_scatter(xb, idx_ref, af_b, None, r_ref[idx_ref], 1.0, O.GATE_XMOD)
        sel = np.zeros(w.T, bool)
        sel[idx_ref] = True
        np.testing.assert_array_equal(got[~sel], xb[~sel])
        U.assert_close(got[sel], ref[sel], "bf16", f"scatter seq {b}", stored_ref=got[sel])


def _full_stack(X, w, check_layers, seqs):
    layers, kinds, bias, x, dev, abi = _setup(X, w)
    mask = _row_mask(w, seqs)
    xd, dm, ws = _teacher_forced(X, w, layers, kinds, bias, x, abi, check_layers, row_mask=mask)
    xs = to_dev(x, w.dtype)
    X.stack_fwd(dm, w.K, w.A, w.N0, w.N1, w.gate, abi, xs,
                torch.from_numpy(bias).cuda() if bias is not None else None, ws)
    assert X.sync_status(ws) == X.OK
    assert torch.equal(xs.view(torch.int16), xd.view(torch.int16))


def test_mod_full_size_sampled(X):
    """Original MoD, ([Sparse(8)] + [Dense]) x 4 with Eq. 6 gating at full size: the first
    and last sparse and dense layers, sampled rows of two sequences."""
    w = I.WORKLOADS["mod_bf16"]
    _full_stack(X, w, {0, 1, 6, 7}, (0, w.B - 1))


def test_a3k16_full_size_sampled(X):
    """X-MoD A3K16 stack, N0=2, N1=2, 48 Sparse(16) layers per block (100 layers) at full
    size: the first dense layer, the first, a middle and the last sparse layer of each
    block, both anchors, sampled rows of two sequences."""
    w = I.WORKLOADS["a3k16_bf16"]
    _full_stack(X, w, {0, 2, 25, 49, 50, 51, 98, 99}, (0, w.B - 1))
