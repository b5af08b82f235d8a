"""Host-side checks of the C ABI that need no GPU: the library builds and loads,
exports every entry point include/xmod.h declares, and rejects bad arguments
before touching the device."""
import ctypes
import os
import re

import pytest

from sparse_depth_token_gb300 import xmod as X

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "xmod.h")


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"XMOD_API\s+[\w\s\*]*?\b(xmod_\w+)\s*\(", src)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(X.EXPORTS)


def test_library_exports_every_declared_symbol():
    L = X.load()
    for name in declared_functions():
        assert hasattr(L, name), name
    out = os.popen(f"nm -D --defined-only {X.library_path()}").read()
    exported = set(re.findall(r" T (\w+)", out))
    assert set(declared_functions()) <= exported
    assert all(s.startswith("xmod_") for s in exported), "internal symbols leak from the library"


def test_noalloc_limit_matches_the_header():
    """The binding's pre-check of the allocation-free entry point uses the header's limit."""
    m = re.search(r"#define\s+XMOD_NOALLOC_MAX_TOKENS\s+\(([^)]*)\)", open(HEADER).read())
    assert m, "XMOD_NOALLOC_MAX_TOKENS not found in the header"
    assert eval(m.group(1), {"__builtins__": {}}) == X.NOALLOC_MAX_TOKENS


def test_version_and_status_strings():
    assert "sm_103a" in X.version()
    for st in (0, -1, -2, -3, -4, -5, -6):
        assert X.status_string(st) != "unknown status"
    assert X.status_string(42) == "unknown status"


def _dims(**kw):
    base = dict(B=2, T=64, d=128, n_heads=4, n_kv_heads=2, head_dim=32, d_ff=352, dtype=X.FP32)
    base.update(kw)
    return X.dims(**base)


def test_workspace_bytes_rules():
    assert X.workspace_bytes(_dims(), 4) > 0
    assert X.workspace_bytes(_dims(d=100), 4) == 0        # d % 8
    assert X.workspace_bytes(_dims(n_kv_heads=3), 4) == 0  # heads % kv heads
    assert X.workspace_bytes(_dims(), 0) == 0
    assert X.workspace_bytes(_dims(), 65) == 0             # K > T
    assert X.workspace_bytes(_dims(dtype=7), 4) == 0
    # bf16 halves the element size of the block scratch; its layouts also hold the
    # tensor-core GEMMs' stream-K scratch: 192 partial tiles of 128 x 256 fp32 and flags
    sk = 192 * 128 * 256 * 4 + 1024
    assert X.workspace_bytes(_dims(dtype=X.BF16), 4) - sk < X.workspace_bytes(_dims(), 4)


FAKE = 0x10000  # 16-byte aligned non-null value; never dereferenced (rejected first)


def _expect(status_fn, code):
    with pytest.raises(X.XmodError) as e:
        status_fn()
    assert e.value.status == code


def test_invalid_arguments_rejected_before_launch():
    dm = _dims()
    ws = FAKE
    L = X.load()
    dmp = ctypes.byref(dm)
    # bad K, bad dims, unaligned or null pointers: nothing reaches CUDA
    assert L.xmod_router_topk(dmp, 0, FAKE, FAKE, None, None, None, FAKE, None, ws, 1 << 30, None) == X.ERR_INVALID_ARG
    assert L.xmod_router_topk(ctypes.byref(_dims(d=12)), 4, FAKE, FAKE, None, None, None, FAKE, None, ws, 1 << 30, None) == X.ERR_INVALID_ARG
    assert L.xmod_router_topk(dmp, 4, FAKE + 4, FAKE, None, None, None, FAKE, None, ws, 1 << 30, None) == X.ERR_INVALID_ARG
    assert L.xmod_router_topk(dmp, 4, None, FAKE, None, None, None, FAKE, None, ws, 1 << 30, None) == X.ERR_INVALID_ARG
    assert L.xmod_router_topk(dmp, 4, FAKE, FAKE, None, None, None, FAKE, None, ws, 16, None) == X.ERR_WORKSPACE
    assert L.xmod_topk(dmp, 4, FAKE, None, None, ws, 1 << 30, None) == X.ERR_INVALID_ARG
    assert L.xmod_gather(dmp, 4, FAKE, FAKE, FAKE + 8, None, None) == X.ERR_INVALID_ARG
    assert L.xmod_gather(dmp, 4, FAKE, FAKE, FAKE, FAKE + 2, None) == X.ERR_INVALID_ARG   # misaligned status
    assert L.xmod_gated_scatter(dmp, 4, FAKE, FAKE, FAKE, FAKE, None, ctypes.c_float(1.0), X.GATE_MOD, None, None) == X.ERR_INVALID_ARG
    assert L.xmod_gated_scatter(dmp, 4, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_float(1.0), 5, None, None) == X.ERR_INVALID_ARG
    w = X.LayerWeights(*([FAKE] * 10), 1.0)
    w_bad = X.LayerWeights(*([FAKE] * 9 + [None]), 1.0)
    assert L.xmod_layer_fwd(dmp, X.LAYER_SPARSE, 4, X.GATE_XMOD, ctypes.byref(w_bad), FAKE, None, None, None, ws, 1 << 30, None) == X.ERR_INVALID_ARG
    assert L.xmod_layer_fwd(dmp, 9, 4, X.GATE_XMOD, ctypes.byref(w), FAKE, None, None, None, ws, 1 << 30, None) == X.ERR_INVALID_ARG
    assert L.xmod_layer_fwd(ctypes.byref(_dims(head_dim=48, d=96, d_ff=96)), X.LAYER_DENSE, 1, X.GATE_XMOD, ctypes.byref(w), FAKE, None, None, None, ws, 1 << 30, None) == X.ERR_UNSUPPORTED
    assert L.xmod_block_fwd(dmp, 0, FAKE, None, ctypes.byref(w), FAKE, FAKE, ws, 1 << 30, None) == X.ERR_INVALID_ARG
    arr = (X.LayerWeights * 6)(*([w] * 6))
    # Eq. 3 layer count must match: N0 + N1 (AK + 1) = 1 + 1 * 5 = 6
    assert L.xmod_stack_fwd(dmp, 4, ctypes.c_double(1.0), 1, 1, X.GATE_XMOD, arr, 5, FAKE, None, ws, 1 << 30, None) == X.ERR_INVALID_ARG
    assert L.xmod_stack_fwd(dmp, 4, ctypes.c_double(0.3), 1, 1, X.GATE_XMOD, arr, 6, FAKE, None, ws, 1 << 30, None) == X.ERR_INVALID_ARG
    assert L.xmod_stack_fwd(dmp, 4, ctypes.c_double(1.0), 1, 1, X.GATE_XMOD, arr, 6, FAKE, None, FAKE + 1, 1 << 30, None) == X.ERR_WORKSPACE
    # the Python binding raises on a negative status
    _expect(lambda: X.gather(dm, 0, FAKE, FAKE, FAKE, stream=0), X.ERR_INVALID_ARG)
    big = _dims(T=64 * 1024, B=1)
    assert L.xmod_topk(ctypes.byref(big), 4, FAKE, FAKE, None, ws, 1 << 40, None) == X.ERR_UNSUPPORTED


def test_backward_arguments_rejected_before_launch():
    """xmod_layer_bwd / xmod_stack_bwd / the wait self-test check their arguments on the
    host: an unknown kind, aliasing outputs, a missing gradient of a weight the kind uses,
    a bad layer count or a short workspace return before anything reaches the device --
    and every layer kind, the Selected-Q / full-KV control included, passes the kind
    check (it reaches the workspace check)."""
    L = X.load()
    dm = _dims()
    dmp = ctypes.byref(dm)
    w = X.LayerWeights(*([FAKE] * 10), 1.0)
    grads = X.LayerGrads(*([FAKE] * 12), None, None)
    A, B, C = FAKE, FAKE + 0x1000, FAKE + 0x2000   # x, dy, dx

    def bwd(kind, x=A, dy=B, dx=C, g=grads, ws_bytes=16):
        return L.xmod_layer_bwd(dmp, kind, 4, X.GATE_XMOD, ctypes.byref(w), x, None, dy,
                                ctypes.c_float(0.0), dx, ctypes.byref(g), FAKE, ws_bytes, None)

    assert bwd(9) == X.ERR_INVALID_ARG
    assert bwd(X.LAYER_SPARSE, dx=A) == X.ERR_INVALID_ARG          # dx aliases x
    assert bwd(X.LAYER_SPARSE, dx=B) == X.ERR_INVALID_ARG          # dx aliases dy
    for kind in (X.LAYER_DENSE, X.LAYER_SPARSE, X.LAYER_ATTN, X.LAYER_ROUTED_FFN,
                 X.LAYER_SPARSE_FULLKV):
        assert bwd(kind) == X.ERR_WORKSPACE, kind
    no_wk = X.LayerGrads(*([FAKE] * 3 + [None] + [FAKE] * 8), None, None)
    assert bwd(X.LAYER_SPARSE_FULLKV, g=no_wk) == X.ERR_INVALID_ARG   # W_k's gradient needed
    assert bwd(X.LAYER_ROUTED_FFN, g=no_wk) == X.ERR_WORKSPACE        # not used: may be NULL
    arr = (X.LayerWeights * 6)(*([w] * 6))
    garr = (X.LayerGrads * 6)(*([grads] * 6))
    assert L.xmod_stack_bwd(dmp, 4, ctypes.c_double(1.0), 1, 1, X.GATE_XMOD, arr, 5, A, None, B,
                            ctypes.c_float(0.0), C, garr, FAKE + 0x10000, FAKE, 1 << 30,
                            None) == X.ERR_INVALID_ARG   # Eq. 3: 1 + 1 * 5 = 6 layers
    assert L.xmod_selftest_wait_timeout(None, 256, None) == X.ERR_INVALID_ARG
    assert L.xmod_selftest_wait_timeout(FAKE, 128, None) == X.ERR_INVALID_ARG
    assert L.xmod_selftest_wait_timeout(FAKE + 4, 256, None) == X.ERR_INVALID_ARG
