"""CPU oracle for the X-MoD / MoD sparse-depth layer forward pass.

TEST INFRASTRUCTURE. Only tests/, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. The CUDA library and its Python binding never import it.

The numerics live in ``xmod_oracle.cpp`` (plain double-precision loops); this
module only marshals numpy arrays into it. The layer-structure arithmetic of
Eq. 2-5 and Eq. 34-36 lives in ``oracle.structure``.
"""
import ctypes
import os

import numpy as np

from . import build as _build

# ATTN / RFFN: the Routed-FFN control's halves; FULLKV: the Selected-Q / full-KV control
DENSE, SPARSE, ATTN, RFFN, FULLKV = 0, 1, 2, 3, 4
GATE_XMOD, GATE_MOD = 0, 1
OK, BAD_ARG, NONFINITE = 0, -1, -5


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("d", ctypes.c_int),
                ("hq", ctypes.c_int), ("hkv", ctypes.c_int), ("hd", ctypes.c_int),
                ("F", ctypes.c_int), ("eps", ctypes.c_double)]


_DP = ctypes.POINTER(ctypes.c_double)
_IP = ctypes.POINTER(ctypes.c_int32)


class LayerW(ctypes.Structure):
    _fields_ = [(n, _DP) for n in ("w_r", "g1", "wq", "wk", "wv", "wo", "g2", "wg", "wu", "wd")] + [
        ("varsigma", ctypes.c_double), ("gq", _DP), ("gk", _DP), ("rope_theta", ctypes.c_double)]


class LayerGrad(ctypes.Structure):
    _fields_ = [(n, _DP) for n in ("w_r", "g1", "wq", "wk", "wv", "wo", "g2", "wg", "wu", "wd")] + [
        ("varsigma", ctypes.c_double), ("gq", _DP), ("gk", _DP)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_round_bf16.restype = ctypes.c_double
        L.oracle_round_bf16.argtypes = [ctypes.c_double]
        L.oracle_round_bf16_n.argtypes = [ctypes.c_int64, _DP]
        L.oracle_router.argtypes = [ctypes.c_int64, ctypes.c_int, _DP, _DP, _DP, _DP, _DP]
        L.oracle_topk.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _DP, _IP]
        L.oracle_rmsnorm.argtypes = [ctypes.c_int64, ctypes.c_int, _DP, _DP, ctypes.c_double, _DP]
        L.oracle_linear.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, _DP, _DP, _DP]
        L.oracle_attention_rows.argtypes = [ctypes.c_int] * 4 + [_DP, _DP, _DP, _DP, _IP, ctypes.c_int]
        L.oracle_block_rows.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, _DP,
                                        ctypes.POINTER(LayerW), _IP, ctypes.c_int, _DP, _DP]
        L.oracle_block_rows_pos.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, _DP,
                                            ctypes.POINTER(LayerW), _IP, ctypes.c_int, _DP, _DP,
                                            _IP]
        L.oracle_qk_transform.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _DP, _DP,
                                          ctypes.c_double, ctypes.c_double, _IP]
        L.oracle_layer_fwd.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.POINTER(LayerW), _DP, _DP, _DP,
                                       _DP, _DP, _IP, _DP, _IP, _IP]
        L.oracle_gated_scatter.argtypes = [ctypes.c_int64, ctypes.c_int, _DP,
                                           ctypes.POINTER(ctypes.c_int64), _DP, _DP, _DP,
                                           ctypes.c_double, ctypes.c_int]
        L.oracle_stack_fwd.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                       ctypes.POINTER(LayerW), _DP, _DP, ctypes.c_int, _IP]
        L.oracle_stack_dyn.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                       ctypes.POINTER(LayerW), _DP, _DP, ctypes.c_double,
                                       ctypes.c_int, _IP, _DP, ctypes.c_int, _IP]
        L.oracle_layer_threshold.argtypes = [ctypes.POINTER(Dims), ctypes.c_int,
                                             ctypes.POINTER(LayerW), _DP, _DP, _DP, _DP, _IP]
        L.oracle_layer_bwd.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.POINTER(LayerW), _DP, _DP, _IP, _DP,
                                       ctypes.c_double, _DP, ctypes.POINTER(LayerGrad), _IP, _DP]
        _lib = L
    return _lib


def num_threads() -> int:
    return lib().oracle_num_threads()


def set_num_threads(n: int) -> None:
    lib().oracle_set_num_threads(int(n))


def _d(a):
    """Contiguous float64 view (or None) and its ctypes pointer."""
    if a is None:
        return None, None
    a = np.ascontiguousarray(a, dtype=np.float64)
    return a, a.ctypes.data_as(_DP)


def _i(a):
    if a is None:
        return None, None
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(_IP)


def _check(st):
    if st != OK:
        raise ValueError(f"oracle returned status {st}")


def round_bf16(v: float) -> float:
    return lib().oracle_round_bf16(float(v))


def round_bf16_array(v):
    """round_bf16 of every element; returns a new float64 array of v's shape."""
    out = np.array(v, dtype=np.float64, copy=True, order="C")
    lib().oracle_round_bf16_n(out.size, out.ctypes.data_as(_DP))
    return out


def router(x, w_r, bias=None):
    """Eq. 8: logits s = x.w_r + bias and gates r = sigmoid(s). x [..., d]."""
    x, xp = _d(x)
    w_r, wp = _d(w_r)
    d = x.shape[-1]
    rows = x.size // d
    bias, bp = _d(None if bias is None else np.reshape(bias, (rows,)))
    s = np.empty(rows)
    r = np.empty(rows)
    lib().oracle_router(rows, d, xp, wp, bp, s.ctypes.data_as(_DP), r.ctypes.data_as(_DP))
    return s.reshape(x.shape[:-1]), r.reshape(x.shape[:-1])


def topk(s, k):
    """Per-sequence top-k of s [B, T]; ties to the lower position; ascending positions."""
    s, sp = _d(np.atleast_2d(s))
    B, T = s.shape
    idx = np.empty((B, k), dtype=np.int32)
    _check(lib().oracle_topk(B, T, k, sp, idx.ctypes.data_as(_IP)))
    return idx


def rmsnorm(x, gamma, eps):
    x, xp = _d(x)
    gamma, gp = _d(gamma)
    d = x.shape[-1]
    out = np.empty_like(x)
    lib().oracle_rmsnorm(x.size // d, d, xp, gp, float(eps), out.ctypes.data_as(_DP))
    return out


def linear(x, W):
    """y = x W^T with W [out, in]."""
    x, xp = _d(x)
    W, wp = _d(W)
    out_f, in_f = W.shape
    rows = x.size // in_f
    y = np.empty((rows, out_f))
    lib().oracle_linear(rows, in_f, out_f, xp, wp, y.ctypes.data_as(_DP))
    return y.reshape(x.shape[:-1] + (out_f,))


def attention(q, k, v, hq, hkv, hd, rows=None):
    """Causal GQA attention on one sequence. q [n, hq*hd], k/v [n, hkv*hd]."""
    q, qp = _d(q)
    k, kp = _d(k)
    v, vp = _d(v)
    n = q.shape[0]
    rows_a, rp = _i(rows)
    nr = n if rows is None else len(rows_a)
    o = np.empty((nr, hq * hd))
    lib().oracle_attention_rows(n, hq, hkv, hd, qp, kp, vp, o.ctypes.data_as(_DP), rp, nr)
    return o


def gated_scatter(x, rows, a, f, r, varsigma, gate):
    """Eq. 7 / Eq. 6 residual written into rows of x [R, d] (returns a new array)."""
    x = np.array(x, dtype=np.float64, copy=True, order="C")
    rows_a = np.ascontiguousarray(rows, dtype=np.int64)
    a, ap = _d(a)
    f_a, fp = _d(f)
    r, rp = _d(r)
    lib().oracle_gated_scatter(len(rows_a), x.shape[-1], x.ctypes.data_as(_DP),
                               rows_a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), ap, fp, rp,
                               float(varsigma), int(gate))
    return x


class Layer:
    """Double-precision weights of one layer, kept alive for the ctypes struct."""

    NAMES = ("w_r", "g1", "wq", "wk", "wv", "wo", "g2", "wg", "wu", "wd")

    def __init__(self, arrays: dict, varsigma: float = 1.0):
        self.arrays = {n: np.ascontiguousarray(arrays[n], dtype=np.float64) for n in self.NAMES}
        # optional Qwen3-style attention extras: QK-norm gains [hd] and the rotary base
        for n in ("gq", "gk"):
            if arrays.get(n) is not None:
                self.arrays[n] = np.ascontiguousarray(arrays[n], dtype=np.float64)
        self.varsigma = float(varsigma)
        self.rope_theta = float(arrays.get("rope_theta", 0.0) or 0.0)
        opt = [self.arrays[n].ctypes.data_as(_DP) if n in self.arrays else None for n in ("gq", "gk")]
        self.struct = LayerW(*[self.arrays[n].ctypes.data_as(_DP) for n in self.NAMES],
                             self.varsigma, *opt, self.rope_theta)


def qk_transform(x, heads, hd, gain=None, eps=1e-6, theta=0.0, pos=None):
    """QK-norm (gain) and rotary embedding (theta) of x [rows, heads * hd]; returns a copy."""
    x = np.array(x, dtype=np.float64, copy=True, order="C")
    g_a, gp = _d(gain)
    p_a, pp = _i(pos)
    lib().oracle_qk_transform(x.shape[0], heads, hd, x.ctypes.data_as(_DP), gp, eps, theta, pp)
    return x


def dims(B, T, d, hq, hkv, hd, F, eps=1e-6) -> Dims:
    return Dims(B, T, d, hq, hkv, hd, F, eps)


def block(dm: Dims, xs, layer: Layer, rows=None, pos=None):
    """Block on one sequence's compact buffer xs [n, d] -> (a, f) for the requested rows.
    pos [n]: original positions of the compact rows (rotary embedding only)."""
    xs, xp = _d(xs)
    n = xs.shape[0]
    rows_a, rp = _i(rows)
    pos_a, pp = _i(pos)
    nr = n if rows is None else len(rows_a)
    a = np.empty((nr, dm.d))
    f = np.empty((nr, dm.d))
    lib().oracle_block_rows_pos(ctypes.byref(dm), n, xp, ctypes.byref(layer.struct), rp, nr,
                                a.ctypes.data_as(_DP), f.ctypes.data_as(_DP), pp)
    return a, f


def layer_fwd(dm: Dims, kind, K, gate, layer: Layer, x, bias=None, idx_force=None,
              row_mask=None):
    """One layer on x [B, T, d]. Returns dict(y, s, r, idx, r_sel) (s..r_sel sparse only)."""
    x, xp = _d(x)
    B, T, d = dm.B, dm.T, dm.d
    assert x.shape == (B, T, d)
    bias_a, bp = _d(bias)
    y = np.empty_like(x)
    out = {"y": y}
    args = [None] * 4
    if kind in (SPARSE, RFFN, FULLKV):
        n = T // K
        out["s"] = np.empty((B, T))
        out["r"] = np.empty((B, T))
        out["idx"] = np.empty((B, n), dtype=np.int32)
        out["r_sel"] = np.empty((B, n))
        args = [out["s"].ctypes.data_as(_DP), out["r"].ctypes.data_as(_DP),
                out["idx"].ctypes.data_as(_IP), out["r_sel"].ctypes.data_as(_DP)]
    f_a, fp = _i(idx_force)
    m_a, mp = _i(row_mask)
    _check(lib().oracle_layer_fwd(ctypes.byref(dm), kind, K, gate, ctypes.byref(layer.struct),
                                  xp, bp, y.ctypes.data_as(_DP), *args, fp, mp))
    return out


def layer_bwd(dm: Dims, kind, K, gate, layer: Layer, x, dy, bias=None, idx_force=None,
              route_coef=0.0):
    """Backward of one layer (DENSE, SPARSE, the FullAttn / Routed-FFN halves ATTN, RFFN,
    or the Selected-Q / full-KV control FULLKV) for the objective sum(dy * y) + route_coef
    * L_route (Eq. 9 on the layer's top-(T/K) decisions), the selection held fixed.
    Returns dict(dx, grads {name: array shaped as the weight}, varsigma, route_loss, idx)."""
    x, xp = _d(x)
    dy, gp = _d(dy)
    B, T, d = dm.B, dm.T, dm.d
    assert x.shape == (B, T, d) and dy.shape == (B, T, d)
    bias_a, bp = _d(bias)
    f_a, fp = _i(idx_force)
    qw, kw = dm.hq * dm.hd, dm.hkv * dm.hd
    shapes = {"w_r": (d,), "g1": (d,), "wq": (qw, d), "wk": (kw, d), "wv": (kw, d),
              "wo": (d, qw), "g2": (d,), "wg": (dm.F, d), "wu": (dm.F, d), "wd": (d, dm.F)}
    for k in ("gq", "gk"):   # QK-norm gains, when the layer has them
        if k in layer.arrays:
            shapes[k] = (dm.hd,)
    grads = {k: np.zeros(v) for k, v in shapes.items()}
    main = ("w_r", "g1", "wq", "wk", "wv", "wo", "g2", "wg", "wu", "wd")
    gs = LayerGrad(*[grads[k].ctypes.data_as(_DP) for k in main], 0.0,
                   *[grads[k].ctypes.data_as(_DP) if k in grads else None for k in ("gq", "gk")])
    dx = np.empty_like(x)
    routed = kind in (SPARSE, RFFN, FULLKV)
    n = T // K if routed else 1
    idx = np.zeros((B, n), np.int32)
    loss = ctypes.c_double(0.0)
    _check(lib().oracle_layer_bwd(ctypes.byref(dm), kind, K, gate, ctypes.byref(layer.struct),
                                  xp, bp, fp, gp, float(route_coef), dx.ctypes.data_as(_DP),
                                  ctypes.byref(gs), idx.ctypes.data_as(_IP), ctypes.byref(loss)))
    return {"dx": dx, "grads": grads, "varsigma": gs.varsigma, "route_loss": loss.value,
            "idx": idx if routed else None}


TOPK, THRESHOLD = 0, 1


def stack_dyn(dm: Dims, K, gate, kinds, layers, x, bias=None, bias_step=0.0,
              mirror_bf16=False, routing=TOPK):
    """Whole stack with the token-choice bias dynamics (X-MoD notes, Eq. 8 and the
    paragraph after it): a sparse layer's logit is w_r.x + bias - bias_step * (times
    the token was selected since the last dense layer). routing TOPK selects T/K per
    sequence, THRESHOLD every token with logit >= 0 (X-MoD notes, causal threshold
    rule at evaluation). Returns (x, idx, s, mask): the final stream and, per sparse
    layer in order, its selection [B, n] (top-k only, else None), logits [B, T] and
    decisions [B, T] (bool)."""
    x = np.array(x, dtype=np.float64, copy=True, order="C")
    bias_a, bp = _d(bias)
    n_sparse = sum(1 for k in kinds if k in (SPARSE, RFFN, FULLKV))
    n = dm.T // K if routing == TOPK else 1
    idx = np.zeros((max(n_sparse, 1), dm.B, n), np.int32)
    s = np.zeros((max(n_sparse, 1), dm.B, dm.T), np.float64)
    mask = np.zeros((max(n_sparse, 1), dm.B, dm.T), np.int32)
    kinds_a = (ctypes.c_int * len(kinds))(*kinds)
    arr = (LayerW * len(layers))(*[l.struct for l in layers])
    _check(lib().oracle_stack_dyn(ctypes.byref(dm), K, gate, len(kinds), kinds_a, arr,
                                  x.ctypes.data_as(_DP), bp, ctypes.c_double(bias_step),
                                  int(bool(mirror_bf16)),
                                  idx.ctypes.data_as(_IP) if routing == TOPK else None,
                                  s.ctypes.data_as(_DP), int(routing), mask.ctypes.data_as(_IP)))
    return (x, idx[:n_sparse] if routing == TOPK else None, s[:n_sparse],
            mask[:n_sparse].astype(bool))


def layer_threshold(dm: Dims, gate, layer, x, bias=None):
    """One sparse layer under the causal threshold rule; returns (y, s, mask)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    s = np.empty((dm.B, dm.T), np.float64)
    mask = np.empty((dm.B, dm.T), np.int32)
    bias_a, bp = _d(bias)
    _check(lib().oracle_layer_threshold(ctypes.byref(dm), gate, ctypes.byref(layer.struct),
                                        x.ctypes.data_as(_DP), bp, y.ctypes.data_as(_DP),
                                        s.ctypes.data_as(_DP), mask.ctypes.data_as(_IP)))
    return y, s, mask.astype(bool)


def stack_fwd(dm: Dims, K, gate, kinds, layers, x, bias=None, mirror_bf16=False,
              seq_mask=None):
    """Whole stack; returns the final residual stream (a new array)."""
    x = np.array(x, dtype=np.float64, copy=True, order="C")
    bias_a, bp = _d(bias)
    kinds_a = (ctypes.c_int * len(kinds))(*kinds)
    arr = (LayerW * len(layers))(*[l.struct for l in layers])
    m_a, mp = _i(seq_mask)
    _check(lib().oracle_stack_fwd(ctypes.byref(dm), K, gate, len(kinds), kinds_a, arr,
                                  x.ctypes.data_as(_DP), bp, int(bool(mirror_bf16)), mp))
    return x
