"""GPU-side helpers of the parity tests: moving seeded inputs to the device and
packing layer weights for the C ABI."""
from __future__ import annotations

import numpy as np
import pytest

import oracle as O
from sparse_depth_token_gb300 import inputs as I

torch = pytest.importorskip("torch")

ABI_NAMES = {"w_r": "w_router", "g1": "rms1", "wq": "wq", "wk": "wk", "wv": "wv", "wo": "wo",
             "g2": "rms2", "wg": "w_gate", "wu": "w_up", "wd": "w_down",
             "gq": "q_norm", "gk": "k_norm"}


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def to_dev(a: np.ndarray, dtype: str):
    """Storage array (bf16 bit patterns or float32) -> device tensor of that dtype."""
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.cuda()


def from_dev(t, dtype: str) -> np.ndarray:
    """Device tensor -> exact float64 numpy copy."""
    if dtype == "bf16":
        bits = t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
        return I.bf16_bits_to_f32(bits).astype(np.float64)
    return t.detach().cpu().numpy().astype(np.float64)


def dev_layer(arrs: dict, dtype: str):
    """Device tensors of one layer, keyed by the C ABI names."""
    return {ABI_NAMES[k]: to_dev(v, dtype) for k, v in arrs.items() if k in ABI_NAMES}


def oracle_layer(arrs: dict, dtype: str) -> O.Layer:
    d = {k: I.to_f64(v, dtype) for k, v in arrs.items() if k in ABI_NAMES}
    if arrs.get("rope_theta"):
        d["rope_theta"] = float(arrs["rope_theta"])
    return O.Layer(d, arrs["varsigma"])


def xmod_dims(w: I.Workload, **over):
    from sparse_depth_token_gb300 import xmod as X
    p = dict(B=w.B, T=w.T, d=w.d, n_heads=w.hq, n_kv_heads=w.hkv, head_dim=w.hd, d_ff=w.F,
             dtype=X.BF16 if w.dtype == "bf16" else X.FP32, rms_eps=w.eps)
    p.update(over)
    return X.dims(**p)


def oracle_dims(w: I.Workload, **over):
    p = dict(B=w.B, T=w.T, d=w.d, hq=w.hq, hkv=w.hkv, hd=w.hd, F=w.F, eps=w.eps)
    p.update(over)
    return O.dims(**p)


def workspace(dm, K):
    from sparse_depth_token_gb300 import xmod as X
    nbytes = X.workspace_bytes(dm, K)
    assert nbytes > 0
    return torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
