"""The bench's algorithmic work -- the numerators of its roofline fractions -- against
closed forms restated here from the block's definition (X-MoD notes, "backbone
configuration": GQA attention, RMSNorm, SwiGLU FFN; Eq. 3 for the layer order), not from
the bench's own code:
  sparse layer (M = B*T/K selected rows, n = T/K per sequence, causal attention):
    2 M d (hq + 2 hkv) hd + 2 M hq hd d + 6 M d F + 2 B n^2 hd hq  FLOPs
  dense layer: the same with M = B*T, n = T;
  routing microbench: x read once by the router (B T d bytes of bf16), the gather's rows
    read and written (2 M d), the scatter's a+f and x rows read and x rows written (3 M d),
    plus the small logit, index and gate arrays;
  backward step: the recomputed forward, two GEMMs per projection (activation and weight
    gradients, each as many FLOPs as the projection), five causal products per head in
    the attention backward."""
import pytest

import bench
from sparse_depth_token_gb300 import inputs as I


def _layers(w):
    ak = int(round(w.A * w.K))
    return ["D"] * w.N0 + (["S"] * ak + ["D"]) * w.N1


def _block_flops(w, M, n):
    qw, kw = w.hq * w.hd, w.hkv * w.hd
    proj = 2 * M * w.d * (qw + 2 * kw) + 2 * M * qw * w.d + 6 * M * w.d * w.F
    att = 2 * w.B * n * n * w.hd * w.hq
    return proj, att


@pytest.mark.parametrize("name,per_sparse_gf,total_tf", [("a4k8_bf16", 212.6, 8.86),
                                                         ("mod_bf16", 386.6, 17.76),
                                                         ("a3k16_bf16", 386.6, 78.34)])
def test_forward_tensor_work(name, per_sparse_gf, total_tf):
    w = I.WORKLOADS[name]
    n = w.T // w.K
    p, a = _block_flops(w, w.B * n, n)
    assert (p + a) / 1e9 == pytest.approx(per_sparse_gf, rel=2e-3)
    total = 0
    for kind in _layers(w):
        p, a = _block_flops(w, w.B * n, n) if kind == "S" else _block_flops(w, w.B * w.T, w.T)
        total += p + a
    assert total / 1e12 == pytest.approx(total_tf, rel=2e-3)
    work = bench.algorithmic_work(w)
    got = sum(v for k, v in work.items() if k in bench.TENSOR_KINDS)
    assert got == pytest.approx(total, rel=1e-12)


@pytest.mark.parametrize("K,gb", [(2, 15.03), (8, 6.98), (16, 5.64)])
def test_routing_bytes(K, gb):
    w = I.WORKLOADS["routing_bf16"]
    BT, M = w.B * w.T, w.B * (w.T // K)
    big = 2 * (BT * w.d + 2 * M * w.d + 3 * M * w.d)   # bf16 rows
    work = bench.routing_work(w, K)
    got = sum(work.values())
    assert big <= got <= big + 16 * (BT + M)            # plus the 4-byte per-token arrays
    assert got / 1e9 == pytest.approx(gb, rel=2e-3)


def test_backward_tensor_work():
    w = I.WORKLOADS["a4k8_bf16"]
    n = w.T // w.K
    want = 0
    for kind in _layers(w):
        M, m = (w.B * n, n) if kind == "S" else (w.B * w.T, w.T)
        p, a = _block_flops(w, M, m)
        want += (p + a) + 2 * p + 2.5 * a   # recompute; dX and dW; S, dP, dQ, dK, dV
    work = bench.backward_work(w)
    got = sum(v for k, v in work.items() if k in bench.BWD_TENSOR_KINDS)
    assert got == pytest.approx(want, rel=1e-12)
