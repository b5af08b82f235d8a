"""Thin Python binding of the C ABI in include/xmod.h (argument marshalling only).

Every function forwards device pointers (torch tensors' data_ptr()) and the
current CUDA stream to libxmod.so; all computation happens in the library's
CUDA kernels. There is no fallback: if the library is missing or fails to load,
load() raises.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

OK = 0
ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE_CHECK, ERR_WORKSPACE = (
    -1, -2, -3, -4, -5, -6)
BF16, FP32 = 0, 1
GATE_XMOD, GATE_MOD = 0, 1
LAYER_DENSE, LAYER_SPARSE, LAYER_ATTN, LAYER_ROUTED_FFN, LAYER_SPARSE_FULLKV = 0, 1, 2, 3, 4

EXPORTS = ("xmod_version", "xmod_status_string", "xmod_workspace_bytes", "xmod_reset_status",
           "xmod_sync_status", "xmod_router_topk", "xmod_topk", "xmod_gather", "xmod_block_fwd",
           "xmod_gated_scatter", "xmod_layer_fwd", "xmod_stack_fwd", "xmod_launch_count",
           "xmod_profile_enable", "xmod_profile_read", "xmod_router_topk_noalloc",
           "xmod_stack_fwd_ex", "xmod_layer_fwd_threshold", "xmod_stack_fwd_sched",
           "xmod_bwd_workspace_bytes", "xmod_layer_bwd", "xmod_stack_bwd_workspace_bytes",
           "xmod_stack_bwd", "xmod_selftest_wait_timeout")

# Largest B*T the allocation-free router entry point accepts (its fixed scratch).
NOALLOC_MAX_TOKENS = 2 * 1024 * 1024


class XmodError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} ({status})")


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("d", ctypes.c_int),
                ("n_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("d_ff", ctypes.c_int), ("dtype", ctypes.c_int),
                ("rms_eps", ctypes.c_float)]


class LayerWeights(ctypes.Structure):
    NAMES = ("w_router", "rms1", "wq", "wk", "wv", "wo", "rms2", "w_gate", "w_up", "w_down")
    _fields_ = [(n, ctypes.c_void_p) for n in NAMES] + [
        ("varsigma", ctypes.c_float), ("q_norm", ctypes.c_void_p), ("k_norm", ctypes.c_void_p),
        ("rope_theta", ctypes.c_float)]


class LayerGrads(ctypes.Structure):
    NAMES = ("w_router", "rms1", "wq", "wk", "wv", "wo", "rms2", "w_gate", "w_up", "w_down",
             "varsigma", "route_loss", "q_norm", "k_norm")
    _fields_ = [(n, ctypes.c_void_p) for n in NAMES]


ROUTE_TOPK, ROUTE_THRESHOLD = 0, 1


class StackOpts(ctypes.Structure):
    _fields_ = [("bias_step", ctypes.c_float), ("layer_stats", ctypes.c_void_p),
                ("update_hist", ctypes.c_void_p), ("routing", ctypes.c_int)]


class KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int),
                ("total_ms", ctypes.c_double)]


_VP = ctypes.c_void_p
_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libxmod.so (building it first if allowed). Raises if unavailable."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path) or not _build.up_to_date():
        if not build_if_missing:
            raise RuntimeError(f"CUDA library not built: {path}")
        _build.build()
    L = ctypes.CDLL(path)
    L.xmod_version.restype = ctypes.c_char_p
    L.xmod_status_string.restype = ctypes.c_char_p
    L.xmod_status_string.argtypes = [ctypes.c_int]
    L.xmod_workspace_bytes.restype = ctypes.c_size_t
    L.xmod_workspace_bytes.argtypes = [ctypes.POINTER(Dims), ctypes.c_int]
    L.xmod_reset_status.argtypes = [_VP, ctypes.c_size_t, _VP]
    L.xmod_sync_status.argtypes = [_VP, _VP]
    L.xmod_router_topk.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, _VP, _VP, _VP, _VP, _VP,
                                   _VP, _VP, _VP, ctypes.c_size_t, _VP]
    L.xmod_topk.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, _VP, _VP, _VP, _VP,
                            ctypes.c_size_t, _VP]
    L.xmod_gather.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, _VP, _VP, _VP, _VP, _VP]
    L.xmod_block_fwd.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, _VP, _VP,
                                 ctypes.POINTER(LayerWeights), _VP, _VP, _VP, ctypes.c_size_t, _VP]
    L.xmod_gated_scatter.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, _VP, _VP, _VP, _VP, _VP,
                                     ctypes.c_float, ctypes.c_int, _VP, _VP]
    L.xmod_layer_fwd.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                 ctypes.POINTER(LayerWeights), _VP, _VP, _VP, _VP, _VP,
                                 ctypes.c_size_t, _VP]
    L.xmod_stack_fwd.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                 ctypes.c_int, ctypes.c_int, ctypes.POINTER(LayerWeights),
                                 ctypes.c_int, _VP, _VP, _VP, ctypes.c_size_t, _VP]
    L.xmod_stack_fwd_ex.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, ctypes.c_double,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.POINTER(LayerWeights), ctypes.c_int, _VP, _VP,
                                    ctypes.POINTER(StackOpts), _VP, ctypes.c_size_t, _VP]
    L.xmod_stack_fwd_sched.argtypes = [ctypes.POINTER(Dims), ctypes.c_int,
                                       ctypes.POINTER(ctypes.c_int32), ctypes.c_int, ctypes.c_int,
                                       ctypes.POINTER(LayerWeights), _VP, _VP,
                                       ctypes.POINTER(StackOpts), _VP, ctypes.c_size_t, _VP]
    L.xmod_layer_fwd_threshold.argtypes = [ctypes.POINTER(Dims), ctypes.c_int,
                                           ctypes.POINTER(LayerWeights), _VP, _VP, _VP, _VP,
                                           ctypes.c_size_t, _VP]
    L.xmod_launch_count.restype = ctypes.c_uint64
    L.xmod_profile_enable.argtypes = [ctypes.c_int]
    L.xmod_profile_read.argtypes = [ctypes.POINTER(KernelTime), ctypes.c_int,
                                    ctypes.POINTER(ctypes.c_int)]
    L.xmod_router_topk_noalloc.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, _VP, _VP, _VP, _VP,
                                           _VP, _VP, _VP]
    L.xmod_selftest_wait_timeout.argtypes = [_VP, ctypes.c_size_t, _VP]
    L.xmod_bwd_workspace_bytes.restype = ctypes.c_size_t
    L.xmod_bwd_workspace_bytes.argtypes = [ctypes.POINTER(Dims), ctypes.c_int]
    L.xmod_layer_bwd.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                 ctypes.POINTER(LayerWeights), _VP, _VP, _VP, ctypes.c_float,
                                 _VP, ctypes.POINTER(LayerGrads), _VP, ctypes.c_size_t, _VP]
    L.xmod_stack_bwd_workspace_bytes.restype = ctypes.c_size_t
    L.xmod_stack_bwd_workspace_bytes.argtypes = [ctypes.POINTER(Dims), ctypes.c_int]
    L.xmod_stack_bwd.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, ctypes.c_double,
                                 ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                 ctypes.POINTER(LayerWeights), ctypes.c_int, _VP, _VP, _VP,
                                 ctypes.c_float, _VP, ctypes.POINTER(LayerGrads), _VP, _VP,
                                 ctypes.c_size_t, _VP]
    _lib = L
    return L


def _p(t):
    """Device pointer of a tensor (None passes NULL). Raw ints pass through."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, st):
    if st != OK:
        raise XmodError(fn, st)


def version() -> str:
    return load().xmod_version().decode()


def status_string(st: int) -> str:
    return load().xmod_status_string(int(st)).decode()


def dims(B, T, d, n_heads, n_kv_heads, head_dim, d_ff, dtype=BF16, rms_eps=1e-6) -> Dims:
    return Dims(B, T, d, n_heads, n_kv_heads, head_dim, d_ff, dtype, rms_eps)


def layer_weights(tensors: dict, varsigma: float = 1.0, rope_theta: float = 0.0) -> LayerWeights:
    """tensors: name -> device tensor for the names of LayerWeights.NAMES, plus the
    optional QK-norm gains "q_norm" / "k_norm" [head_dim]; rope_theta > 0 turns on the
    rotary embedding. The struct keeps a reference to the tensors so their memory
    outlives every call using it."""
    lw = LayerWeights(*[_p(tensors.get(n)) for n in LayerWeights.NAMES], float(varsigma),
                      _p(tensors.get("q_norm")), _p(tensors.get("k_norm")), float(rope_theta))
    lw._keep = dict(tensors)
    return lw


def workspace_bytes(dm: Dims, K: int) -> int:
    return int(load().xmod_workspace_bytes(ctypes.byref(dm), int(K)))


def reset_status(ws, stream=None):
    _check("xmod_reset_status", load().xmod_reset_status(_p(ws), ws.numel() * ws.element_size(),
                                                         _stream(stream)))


def sync_status(ws, stream=None) -> int:
    return int(load().xmod_sync_status(_p(ws), _stream(stream)))


def _wsb(ws):
    return ws.numel() * ws.element_size() if ws is not None else 0


def router_topk(dm, K, x, w_r, bias, logits, r, idx, r_sel, ws, stream=None):
    _check("xmod_router_topk", load().xmod_router_topk(
        ctypes.byref(dm), int(K), _p(x), _p(w_r), _p(bias), _p(logits), _p(r), _p(idx), _p(r_sel),
        _p(ws), _wsb(ws), _stream(stream)))


def topk(dm, K, logits, idx, r_sel, ws, stream=None):
    _check("xmod_topk", load().xmod_topk(ctypes.byref(dm), int(K), _p(logits), _p(idx), _p(r_sel),
                                         _p(ws), _wsb(ws), _stream(stream)))


def gather(dm, K, x, idx, xs, stream=None, status=None):
    """status: None, or a device int32 tensor that receives XMOD_ERR_DEVICE_CHECK when a
    position is out of range or not ascending (that row is skipped)."""
    _check("xmod_gather", load().xmod_gather(ctypes.byref(dm), int(K), _p(x), _p(idx), _p(xs),
                                             _p(status), _stream(stream)))


def block_fwd(dm, n_per_seq, xs, idx, w: LayerWeights, a_out, f_out, ws, stream=None):
    _check("xmod_block_fwd", load().xmod_block_fwd(
        ctypes.byref(dm), int(n_per_seq), _p(xs), _p(idx), ctypes.byref(w), _p(a_out), _p(f_out),
        _p(ws), _wsb(ws), _stream(stream)))


def gated_scatter(dm, K, x, idx, r_sel, a, f, varsigma, gate, stream=None, status=None):
    """status: as for gather (a bad position's row is not written)."""
    _check("xmod_gated_scatter", load().xmod_gated_scatter(
        ctypes.byref(dm), int(K), _p(x), _p(idx), _p(r_sel), _p(a), _p(f), float(varsigma),
        int(gate), _p(status), _stream(stream)))


def layer_fwd(dm, kind, K, gate, w: LayerWeights, x, bias, idx_out, r_sel_out, ws, stream=None):
    _check("xmod_layer_fwd", load().xmod_layer_fwd(
        ctypes.byref(dm), int(kind), int(K), int(gate), ctypes.byref(w), _p(x), _p(bias),
        _p(idx_out), _p(r_sel_out), _p(ws), _wsb(ws), _stream(stream)))


def stack_fwd(dm, K, A, N0, N1, gate, layers, x, bias, ws, stream=None):
    # the array copies the structs; the caller's LayerWeights keep the tensors alive
    arr = (LayerWeights * len(layers))(*layers)
    _check("xmod_stack_fwd", load().xmod_stack_fwd(
        ctypes.byref(dm), int(K), float(A), int(N0), int(N1), int(gate), arr, len(layers), _p(x),
        _p(bias), _p(ws), _wsb(ws), _stream(stream)))


def stack_fwd_ex(dm, K, A, N0, N1, gate, layers, x, bias, ws, bias_step=0.0, layer_stats=None,
                 update_hist=None, routing=ROUTE_TOPK, stream=None):
    """xmod_stack_fwd_ex: the stack with the token-choice bias dynamics (bias_step), the
    selection rule (ROUTE_TOPK or ROUTE_THRESHOLD) and, when given, the routing
    statistics: layer_stats int32 [n_sparse, B, 4] and update_hist int32
    [N1, B, AK + 1] (device tensors)."""
    arr = (LayerWeights * len(layers))(*layers)
    opts = StackOpts(float(bias_step), _p(layer_stats), _p(update_hist), int(routing))
    _check("xmod_stack_fwd_ex", load().xmod_stack_fwd_ex(
        ctypes.byref(dm), int(K), float(A), int(N0), int(N1), int(gate), arr, len(layers), _p(x),
        _p(bias), ctypes.byref(opts), _p(ws), _wsb(ws), _stream(stream)))


def stack_fwd_sched(dm, K, kinds, gate, layers, x, bias, ws, bias_step=0.0, layer_stats=None,
                    update_hist=None, routing=ROUTE_TOPK, stream=None):
    """xmod_stack_fwd_sched: the stack in an explicit layer order (kinds: DENSE / SPARSE
    per layer), e.g. the segment stacks of X-MoD notes Eq. 35 / 36."""
    arr = (LayerWeights * len(layers))(*layers)
    ks = (ctypes.c_int32 * len(kinds))(*[int(k) for k in kinds])
    opts = StackOpts(float(bias_step), _p(layer_stats), _p(update_hist), int(routing))
    _check("xmod_stack_fwd_sched", load().xmod_stack_fwd_sched(
        ctypes.byref(dm), int(K), ks, len(kinds), int(gate), arr, _p(x), _p(bias),
        ctypes.byref(opts), _p(ws), _wsb(ws), _stream(stream)))


def layer_fwd_threshold(dm, gate, w, x, bias, ws, count_out=None, stream=None):
    """xmod_layer_fwd_threshold: one sparse layer under the causal threshold rule;
    count_out (device int32 [B]) receives each sequence's routed token count."""
    _check("xmod_layer_fwd_threshold", load().xmod_layer_fwd_threshold(
        ctypes.byref(dm), int(gate), ctypes.byref(w), _p(x), _p(bias), _p(count_out), _p(ws),
        _wsb(ws), _stream(stream)))


def launch_count() -> int:
    return int(load().xmod_launch_count())


def profile_enable(on: bool) -> None:
    load().xmod_profile_enable(1 if on else 0)


def profile_read(max_kinds: int = 64) -> dict:
    """{kernel kind: (launches, total_ms)} recorded since the last read."""
    arr = (KernelTime * max_kinds)()
    n = ctypes.c_int(0)
    _check("xmod_profile_read", load().xmod_profile_read(arr, max_kinds, ctypes.byref(n)))
    return {arr[i].name.decode(): (arr[i].launches, arr[i].total_ms) for i in range(n.value)}


def router_topk_noalloc(dm, K, x, w_r, bias, idx, r_sel, status=None, stream=None):
    """xmod_router_topk without a workspace, for callers that cannot allocate device
    memory: the library's own fixed scratch holds the logits (B*T <= NOALLOC_MAX_TOKENS).
    `status` (optional device int32 tensor) receives the call's device status."""
    if dm.B * dm.T > NOALLOC_MAX_TOKENS:
        raise XmodError("xmod_router_topk_noalloc", ERR_UNSUPPORTED)
    _check("xmod_router_topk_noalloc", load().xmod_router_topk_noalloc(
        ctypes.byref(dm), int(K), _p(x), _p(w_r), _p(bias), _p(idx), _p(r_sel), _p(status),
        _stream(stream)))


def bwd_workspace_bytes(dm: Dims, K: int) -> int:
    return int(load().xmod_bwd_workspace_bytes(ctypes.byref(dm), int(K)))


def layer_grads(tensors: dict) -> LayerGrads:
    """LayerGrads from fp32 device tensors keyed by LayerGrads.NAMES (missing: NULL)."""
    return LayerGrads(*[_p(tensors.get(n)) for n in LayerGrads.NAMES])


def layer_bwd(dm, kind, K, gate, w: LayerWeights, x, bias, dy, route_coef, dx, grads: LayerGrads,
              ws, stream=None):
    """xmod_layer_bwd: dx and the weight gradients of sum(dy * y) + route_coef * L_route."""
    _check("xmod_layer_bwd", load().xmod_layer_bwd(
        ctypes.byref(dm), int(kind), int(K), int(gate), ctypes.byref(w), _p(x), _p(bias), _p(dy),
        float(route_coef), _p(dx), ctypes.byref(grads), _p(ws), _wsb(ws), _stream(stream)))


def stack_bwd_workspace_bytes(dm: Dims, K: int) -> int:
    return int(load().xmod_stack_bwd_workspace_bytes(ctypes.byref(dm), int(K)))


def stack_bwd(dm, K, A, N0, N1, gate, layers, x, bias, dy, route_coef, dx, grads, checkpoints,
              ws, stream=None):
    """xmod_stack_bwd: the Eq. 3 stack's backward; grads is a list of LayerGrads (one per
    layer), checkpoints a device buffer [n_layers, B, T, d]."""
    arr = (LayerWeights * len(layers))(*layers)
    garr = (LayerGrads * len(grads))(*grads)
    _check("xmod_stack_bwd", load().xmod_stack_bwd(
        ctypes.byref(dm), int(K), float(A), int(N0), int(N1), int(gate), arr, len(layers), _p(x),
        _p(bias), _p(dy), float(route_coef), _p(dx), garr, _p(checkpoints), _p(ws), _wsb(ws),
        _stream(stream)))


def selftest_wait_timeout(ws, stream=None):
    """xmod_selftest_wait_timeout: one CTA runs the kernels' bounded wait on a barrier
    that nothing completes until it gives up (about 2 s); the status word of ws then holds
    ERR_TIMEOUT."""
    _check("xmod_selftest_wait_timeout",
           load().xmod_selftest_wait_timeout(_p(ws), _wsb(ws), _stream(stream)))
