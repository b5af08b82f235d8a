"""Seeded synthetic inputs for the sparse-depth layer stack.

This module draws random numbers and stores them in the storage dtype; it holds
none of the method's arithmetic. The same arrays feed the CUDA library and the
CPU oracle, so both see bit-identical inputs.

Workloads (shapes and distributions follow the X-MoD notes' backbone table --
GQA, head_dim 128, SwiGLU -- and its sequence lengths of 4k-32k):
  tiny_fp32      fp32, [D] + [S(4)]x4 + [D] with N0=1, N1=1, A=1, K=4 (6 layers),
                 d=128, 4 q / 2 kv heads, hd=32, F=352, B=2, T=64, bias ~ N(0, 0.1^2)
  routing_bf16   bf16 routing microbench, B=64, T=8192, d=4096, K in {2, 8, 16},
                 bias 0, given block output (a+f) ~ N(0, 1)
  mod_bf16       bf16 MoD ([S(8)] + [D]) x 4 (8 layers), Eq. 6, d=2048, 16/4 heads,
                 hd=128, F=5632, B=4, T=8192, seed 1
  a4k8_bf16      bf16 X-MoD A4K8 block: 32 S(8) + 1 D, Eq. 7, d=1536, 12/4 heads,
                 hd=128, F=4096, B=8, T=4096, varsigma ~ U(0.5, 1.5), bias ~ N(0, 0.1^2)
  a3k16_bf16     bf16 X-MoD A3K16 stack: N0=2, N1=2, AK=48, K=16 (100 layers), Eq. 7,
                 d=2048, 16/4 heads, hd=128, F=5632, B=4, T=16384, varsigma ~ U(0.5, 1.5)
Common: x ~ N(0, 1); matrices ~ N(0, 0.02^2); router w_r ~ N(0, 1/d); RMSNorm gains 1.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np

DENSE, SPARSE = 0, 1
GATE_XMOD, GATE_MOD = 0, 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str          # "bf16" or "fp32"
    B: int
    T: int
    d: int
    hq: int
    hkv: int
    hd: int
    F: int
    K: int
    A: float
    N0: int
    N1: int
    n_layers: int       # physical layers (data, not derived here)
    gate: int
    seed: int
    bias_std: float = 0.0          # 0: no bias
    varsigma_range: tuple = (1.0, 1.0)
    eps: float = 1e-6
    weight_std: float = 0.02      # std of the projection matrices

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", "fp32", 2, 64, 128, 4, 2, 32, 352, 4, 1, 1, 1, 6,
                          GATE_XMOD, 0, bias_std=0.1),
    "routing_bf16": Workload("routing_bf16", "bf16", 64, 8192, 4096, 32, 8, 128, 14336, 8,
                             1, 0, 1, 0, GATE_XMOD, 1),
    "mod_bf16": Workload("mod_bf16", "bf16", 4, 8192, 2048, 16, 4, 128, 5632, 8, 0.125, 0, 4,
                         8, GATE_MOD, 1),
    "a4k8_bf16": Workload("a4k8_bf16", "bf16", 8, 4096, 1536, 12, 4, 128, 4096, 8, 4, 0, 1,
                          33, GATE_XMOD, 3, bias_std=0.1, varsigma_range=(0.5, 1.5)),
    "a3k16_bf16": Workload("a3k16_bf16", "bf16", 4, 16384, 2048, 16, 4, 128, 5632, 16, 3, 2,
                           2, 100, GATE_XMOD, 4, varsigma_range=(0.5, 1.5)),
}

_TENSORS = ("w_r", "g1", "wq", "wk", "wv", "wo", "g2", "wg", "wu", "wd")


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns the uint16 bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    rounding = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32)


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 copy of a stored array (bf16 bit patterns or float32)."""
    if dtype == "bf16":
        return bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *key])))


def _normal(seed, key, shape, std, dtype):
    g = _rng(seed, *key)
    a = g.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return f32_to_bf16_bits(a) if dtype == "bf16" else a


def layer_weights(w: Workload, layer: int) -> dict:
    """Weights of one layer in the storage dtype. Matrices are [out, in] row-major."""
    d, hq, hkv, hd, F = w.d, w.hq, w.hkv, w.hd, w.F
    shapes = {"wq": (hq * hd, d), "wk": (hkv * hd, d), "wv": (hkv * hd, d), "wo": (d, hq * hd),
              "wg": (F, d), "wu": (F, d), "wd": (d, F)}
    out = {}
    for t, name in enumerate(_TENSORS):
        key = (1000 + layer, t)
        if name in shapes:
            out[name] = _normal(w.seed, key, shapes[name], w.weight_std, w.dtype)
        elif name == "w_r":
            out[name] = _normal(w.seed, key, (d,), 1.0 / np.sqrt(d), w.dtype)
        else:  # RMSNorm gains
            ones = np.ones(d, dtype=np.float32)
            out[name] = f32_to_bf16_bits(ones) if w.dtype == "bf16" else ones
    lo, hi = w.varsigma_range
    out["varsigma"] = float(_rng(w.seed, 1000 + layer, 99).uniform(lo, hi)) if hi > lo else lo
    return out


def all_layer_weights(w: Workload, n_layers: int | None = None, threads: int | None = None):
    n = w.n_layers if n_layers is None else n_layers
    threads = threads or min(16, os.cpu_count() or 1)
    with _cf.ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(lambda l: layer_weights(w, l), range(n)))


def residual_stream(w: Workload) -> np.ndarray:
    """x [B, T, d] ~ N(0, 1) in the storage dtype (generated per sequence)."""
    def one(b):
        return _normal(w.seed, (1, b), (w.T, w.d), 1.0, w.dtype)
    threads = min(16, os.cpu_count() or 1)
    with _cf.ThreadPoolExecutor(max_workers=threads) as ex:
        rows = list(ex.map(one, range(w.B)))
    return np.stack(rows)


def router_bias(w: Workload):
    """Signed per-token router bias [B, T] as float32, or None when the workload has none."""
    if w.bias_std == 0.0:
        return None
    return _rng(w.seed, 2).standard_normal(size=(w.B, w.T), dtype=np.float32) * np.float32(
        w.bias_std)


def given_block_output(w: Workload, M: int) -> np.ndarray:
    """The routing microbench's stand-in for the block output (a + f) ~ N(0, 1), [M, d]."""
    return _normal(w.seed, (3,), (M, w.d), 1.0, w.dtype)


def shard_sequences(B: int, rank: int, world: int) -> range:
    """Contiguous share of the B sequences for one rank (sequences are independent)."""
    per, extra = divmod(B, world)
    lo = rank * per + min(rank, extra)
    return range(lo, lo + per + (1 if rank < extra else 0))
