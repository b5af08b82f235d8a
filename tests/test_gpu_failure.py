"""Failure detection on the GPU without a fault, a trap or a hang: the kernels' bounded
wait (the helper every tcgen05 kernel waits through) runs out on an mbarrier that nothing
completes; the status word reports ERR_TIMEOUT, the wait says it gave up and raised the
CTA's abort flag, and the same CUDA context then computes normally."""
import time

import numpy as np
import pytest

import oracle as O
from tests._gpu import need_gpu, torch, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def X():
    need_gpu()
    from sparse_depth_token_gb300 import xmod
    xmod.load()
    return xmod


def test_bounded_wait_gives_up_and_the_context_survives(X):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    X.reset_status(ws)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    X.selftest_wait_timeout(ws)
    assert X.sync_status(ws) == X.ERR_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert 1.9 <= elapsed < 60.0, elapsed   # the 2 s limit, then the kernel returned
    words = ws.view(torch.int32).cpu().numpy()
    assert words[1] == 0 and words[2] == 1   # gave up; abort flag raised
    # the context is intact: a top-k on given logits, bit-exact against the oracle
    B, T, K = 2, 1000, 4
    s = np.random.default_rng(8).standard_normal((B, T)).astype(np.float32)
    dm = X.dims(B, T, 8, 1, 1, 8, 8, X.FP32)
    wsk = workspace(dm, K)
    idx = torch.empty((B, T // K), dtype=torch.int32, device="cuda")
    r_sel = torch.empty((B, T // K), dtype=torch.float32, device="cuda")
    X.reset_status(wsk)
    X.topk(dm, K, torch.from_numpy(s).cuda(), idx, r_sel, wsk)
    assert X.sync_status(wsk) == X.OK
    np.testing.assert_array_equal(idx.cpu().numpy(), O.topk(s.astype(np.float64), T // K))


def test_selftest_rejects_a_bad_buffer(X):
    ws = torch.zeros(128, dtype=torch.uint8, device="cuda")   # below 256 bytes
    with pytest.raises(X.XmodError):
        X.selftest_wait_timeout(ws)
