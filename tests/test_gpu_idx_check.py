"""Device-side checks of caller-supplied positions (xmod_gather, xmod_gated_scatter,
xmod_block_fwd): a row whose position is outside [0, T) or not above the previous
row's in its sequence is reported as XMOD_ERR_DEVICE_CHECK, and gather and scatter
write nothing for it.

Every bad position used here still addresses memory inside the stream, so a broken
check could not reach outside the allocation: a duplicated position, a position below
its predecessor, and position T in sequence 0 (the address of sequence 1's first
row). The expected results come from the same kernels run on the valid positions with
the bad rows' outputs taken out by hand, so the comparison is bitwise."""
import numpy as np
import pytest

from sparse_depth_token_gb300 import inputs as I
from tests._gpu import need_gpu, to_dev, torch, workspace, xmod_dims

pytestmark = pytest.mark.gpu

B, T, K, D = 2, 64, 4, 64
N = T // K


@pytest.fixture(scope="module")
def X():
    need_gpu()
    from sparse_depth_token_gb300 import xmod
    xmod.load()
    return xmod


def _positions():
    g = np.random.default_rng(5)
    good = np.stack([np.sort(g.choice(np.arange(1, T), N, replace=False)) for _ in range(B)])
    good = good.astype(np.int32)   # position 0 of sequence 1 is never selected
    bad = good.copy()
    bad[0, 5] = bad[0, 4]          # duplicate
    bad[0, N - 1] = T              # out of range: the address of row (1, 0)
    q = int(np.setdiff1d(np.arange(1, good[1, 2]), good[1])[0])
    bad[1, 3] = q                  # below its predecessor, not selected elsewhere
    bad_rows = [(0, 5), (0, N - 1), (1, 3)]
    return good, bad, bad_rows


def _setup(X):
    w = I.WORKLOADS["routing_bf16"].replace(B=B, T=T, d=D, seed=61)
    dm = xmod_dims(w)
    g = np.random.default_rng(6)
    x = I.f32_to_bf16_bits(g.standard_normal((B, T, D)).astype(np.float32))
    return dm, x


def test_gather_skips_bad_rows(X):
    dm, x = _setup(X)
    good, bad, bad_rows = _positions()
    xd = to_dev(x, "bf16")
    ref = torch.zeros((B * N, D), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    X.gather(dm, K, xd, torch.from_numpy(good).cuda(), ref, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == X.OK
    sentinel = torch.full((B * N, D), 7.0, dtype=torch.bfloat16, device="cuda")
    got = sentinel.clone()
    X.gather(dm, K, xd, torch.from_numpy(bad).cuda(), got, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == X.ERR_DEVICE_CHECK
    want = ref.clone()
    for b, j in bad_rows:
        want[b * N + j] = sentinel[b * N + j]
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("gate", [0, 1])
def test_gated_scatter_skips_bad_rows(X, gate):
    dm, x = _setup(X)
    good, bad, bad_rows = _positions()
    g = np.random.default_rng(7)
    a = g.standard_normal((B * N, D)).astype(np.float32)
    f = g.standard_normal((B * N, D)).astype(np.float32)
    r = g.uniform(0.1, 0.9, (B, N)).astype(np.float32)
    for b, j in bad_rows:           # the reference leaves these rows' positions unchanged
        a[b * N + j] = 0.0
        f[b * N + j] = 0.0
    a0 = g.standard_normal((B * N, D)).astype(np.float32)   # the bad run's own a, f
    f0 = g.standard_normal((B * N, D)).astype(np.float32)
    for m in range(B * N):
        if (m // N, m % N) not in bad_rows:
            a0[m], f0[m] = a[m], f[m]
    ad, fd = to_dev(I.f32_to_bf16_bits(a), "bf16"), to_dev(I.f32_to_bf16_bits(f), "bf16")
    a0d, f0d = to_dev(I.f32_to_bf16_bits(a0), "bf16"), to_dev(I.f32_to_bf16_bits(f0), "bf16")
    rd = torch.from_numpy(r).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    want = to_dev(x, "bf16")
    X.gated_scatter(dm, K, want, torch.from_numpy(good).cuda(), rd, ad, fd, 0.8, gate, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == X.OK
    got = to_dev(x, "bf16")
    X.gated_scatter(dm, K, got, torch.from_numpy(bad).cuda(), rd, a0d, f0d, 0.8, gate, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == X.ERR_DEVICE_CHECK
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    assert torch.equal(got[1, 0].view(torch.int16), to_dev(x, "bf16")[1, 0].view(torch.int16))


def test_block_fwd_reports_bad_rows(X):
    """The block reads clamped positions for bad rows (nothing outside the stream) and
    reports them; with valid positions the same call reports nothing."""
    w = I.WORKLOADS["a4k8_bf16"].replace(B=B, T=T, d=256, hq=4, hkv=2, F=256, seed=62)
    lw = I.layer_weights(w, 0)
    from tests._gpu import dev_layer
    dev = dev_layer(lw, "bf16")
    abi = X.layer_weights(dev, lw["varsigma"])
    dm = xmod_dims(w)
    ws = workspace(dm, K)
    xd = to_dev(I.residual_stream(w), "bf16")
    good, bad, _ = _positions()
    a = torch.empty((B * N, w.d), dtype=torch.bfloat16, device="cuda")
    f = torch.empty_like(a)
    X.reset_status(ws)
    X.block_fwd(dm, N, xd, torch.from_numpy(good).cuda(), abi, a, f, ws)
    assert X.sync_status(ws) == X.OK
    X.reset_status(ws)
    X.block_fwd(dm, N, xd, torch.from_numpy(bad).cuda(), abi, a, f, ws)
    assert X.sync_status(ws) == X.ERR_DEVICE_CHECK
    assert torch.isfinite(a.float()).all() and torch.isfinite(f.float()).all()
