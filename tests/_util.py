"""Shared helpers of the parity tests: tolerances, input preparation, tensor moves.

Tolerances (stated by the method's acceptance bar): bf16 paths max-abs <= 2e-2 and
relative L2 <= 1e-2 against the oracle's unrounded double result; fp32 paths
relative 1e-5 (relative L2 and max|diff| / max|ref|). Indices are bit-exact.
"""
from __future__ import annotations

import numpy as np

import oracle as O
from sparse_depth_token_gb300 import inputs as I

BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 1e-2
FP32_REL = 1e-5
ROUTING_MARGIN = 1e-3       # enforced gap at the k-th rank of generated logits
NEAR_TIE = 1e-4             # band in which a later layer's routing may legitimately differ


def rel_l2(got, ref) -> float:
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def bf16_half_ulp(v) -> np.ndarray:
    """Half the bf16 spacing at |v| (8 significant bits): the storage rounding of a bf16 output."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def assert_close(got, ref, dtype: str, what: str = "", stored_ref=None):
    """bf16: max-abs <= 2e-2 and rel-L2 <= 1e-2; fp32: relative 1e-5.

    stored_ref: for a bf16 output that overwrites a bf16 tensor (the residual
    stream), the values it is stored as; the max-abs bound then applies to the
    arithmetic beyond the output's own storage rounding (half a bf16 spacing at
    |stored_ref|, which by itself exceeds 2e-2 for |y| >= 8)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if dtype == "bf16":
        err = np.abs(got - ref)
        if stored_ref is not None:
            err = np.maximum(err - bf16_half_ulp(stored_ref), 0.0)
        mx = float(np.max(err)) if got.size else 0.0
        rl = rel_l2(got, ref)
        if not (mx <= BF16_MAX_ABS and rl <= BF16_REL_L2):
            i = int(np.argmax(err))
            raise AssertionError(
                f"{what}: max-abs {mx:.3e}, rel-L2 {rl:.3e}; worst element {i}: got "
                f"{got.flat[i]:.6f} ref {ref.flat[i]:.6f}; max|ref| {np.max(np.abs(ref)):.3f}, "
                f"rms(ref) {np.sqrt(np.mean(ref ** 2)):.4f}, count(err>2e-2) "
                f"{int(np.count_nonzero(err > BF16_MAX_ABS))} of {err.size}")
    else:
        rl = rel_l2(got, ref)
        scale = float(np.max(np.abs(ref))) if ref.size else 1.0
        mr = float(np.max(np.abs(got - ref))) / (scale if scale > 0 else 1.0) if got.size else 0.0
        assert rl <= FP32_REL and mr <= FP32_REL, f"{what}: rel-L2 {rl:.3e}, max-rel {mr:.3e}"


# ------------------------------------------------------------------ routing margins

def _bf16_step_down(bits: np.uint16, up: bool) -> np.uint16:
    """Next bf16 value toward +inf (up) or -inf, on the bit pattern."""
    b = int(bits)
    neg = bool(b & 0x8000)
    mag = b & 0x7FFF
    if mag == 0:
        return np.uint16(0x0001 if up else 0x8001)
    if up != neg:            # moving away from zero
        return np.uint16(b + 1)
    return np.uint16(b - 1)


def enforce_routing_margin(x_store, dtype, w_r_store, bias, K, margin=ROUTING_MARGIN):
    """Make the oracle's k-th-rank gap of every sequence at least `margin` by
    demoting non-selected tokens whose logit lies within 2*margin of the k-th:
    the coordinate with the largest |w_r| is moved one storage-precision step at a
    time against the sign of w_r. Returns (new x, number of rows touched)."""
    x = np.array(x_store, copy=True)
    B, T, d = x.shape
    n = T // K
    w64 = I.to_f64(w_r_store, dtype)
    mstar = int(np.argmax(np.abs(w64)))
    up = w64[mstar] < 0          # increasing x lowers the logit when w_r < 0
    touched = 0
    for b in range(B):
        xb64 = I.to_f64(x[b], dtype)
        s, _ = O.router(xb64, w64, None if bias is None else bias[b])
        order = np.lexsort((np.arange(T), -s))
        sel = order[:n]
        kth = s[sel].min()
        for t in order[n:]:
            if s[t] < kth - 2 * margin:
                break
            bt = None if bias is None else np.array([bias[b, t]])
            # jump most of the way, then step in storage precision until the gap holds
            target = I.to_f64(x[b, t, mstar:mstar + 1], dtype)[0] - (
                s[t] - (kth - 1.25 * margin)) / w64[mstar]
            t32 = np.array([target], dtype=np.float32)
            x[b, t, mstar] = I.f32_to_bf16_bits(t32)[0] if dtype == "bf16" else t32[0]
            for _ in range(10000):
                row = I.to_f64(x[b, t], dtype)
                s[t] = O.router(row[None, :], w64, bt)[0][0]
                if s[t] <= kth - margin:
                    break
                if dtype == "bf16":
                    x[b, t, mstar] = _bf16_step_down(x[b, t, mstar], up)
                else:
                    x[b, t, mstar] = np.nextafter(x[b, t, mstar],
                                                  np.float32(np.inf if up else -np.inf))
            assert s[t] <= kth - margin
            touched += 1
    return x, touched


def kth_gap(s, n):
    """Per-sequence gap between the n-th and (n+1)-th largest logits."""
    srt = -np.sort(-np.asarray(s), axis=-1)
    if n >= srt.shape[-1]:
        return np.full(srt.shape[0], np.inf)
    return srt[:, n - 1] - srt[:, n]


def check_selection(idx_gpu, s_oracle, n, band=NEAR_TIE):
    """Accept the GPU's selection if it is a valid top-n of the oracle logits up to
    a `band`-wide near-tie zone: returns the number of sequences that differ from
    the oracle's own choice (0 when bit-exact)."""
    B, T = s_oracle.shape
    ref = O.topk(s_oracle, n)
    differ = 0
    for b in range(B):
        g = np.asarray(idx_gpu[b])
        assert len(g) == n and np.all(np.diff(g) > 0) and g.min() >= 0 and g.max() < T
        if np.array_equal(g, ref[b]):
            continue
        differ += 1
        kth = np.sort(s_oracle[b])[::-1][n - 1]
        chosen = np.zeros(T, bool)
        chosen[g] = True
        assert np.all(s_oracle[b][chosen] >= kth - band), "GPU selected a token below the band"
        assert np.all(s_oracle[b][~chosen] <= kth + band), "GPU skipped a token above the band"
    return differ
