"""Token-choice bias dynamics and routing diagnostics on the CPU (no GPU).

X-MoD notes, Eq. 8 and the paragraph after it: inside a sparse-dense block a token's
bias grows each time it is selected and is cleared at the next dense anchor; the
section "routing diagnostics" and Table 10 define coverage, adjacent-layer Jaccard,
threshold / top-k mask agreement and update counts, with two analytic references.

Pins: the analytic reference columns of Table 10 (tests/golden/table10_reference.json);
the references reproduced by the diagnostics on constructed masks (same subset every
layer: exact; independent random subsets: within sampling error); the oracle stack
with no growth equal to the constant-bias stack; and with an overwhelming growth the
closed-form rotation -- every token exactly once per block when the block has K sparse
layers, each penalised token showing the full penalty in the next layer's logits and
none at the first layer of a block (the anchor cleared it)."""
import json
import os

import numpy as np
import pytest

import oracle as O
from oracle import diagnostics as D
from oracle import structure as S
from sparse_depth_token_gb300 import diagnostics as PD
from sparse_depth_token_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "table10_reference.json")


def test_table10_reference_columns():
    rows = json.load(open(GOLDEN))["rows"]
    for r in rows:
        p, L = 1.0 / r["K"], r["L"]
        cov_s, jac_s, dist_s = D.repeated_subset_reference(p, L)
        cov_r, jac_r, dist_r = D.independent_random_reference(p, L)
        # printed to 4 significant figures
        assert abs(100 * cov_s - r["repeated_coverage"]) < 5e-3, r
        assert abs(100 * jac_s - r["repeated_jaccard"]) < 5e-3, r
        assert abs(100 * cov_r - r["random_coverage"]) < 5e-3, r
        assert abs(100 * jac_r - r["random_jaccard"]) < 5e-4, r
        assert abs(dist_s.sum() - 1) < 1e-12 and abs(dist_r.sum() - 1) < 1e-12
        assert abs((np.arange(L + 1) * dist_r).sum() - L * p) < 1e-9   # Binomial mean


def _repeated_masks(L, B, T, n, g):
    m = np.zeros((L, B, T), bool)
    for b in range(B):
        m[:, b, g.choice(T, n, replace=False)] = True
    return m


def _random_masks(L, B, T, n, g):
    m = np.zeros((L, B, T), bool)
    for l in range(L):
        for b in range(B):
            m[l, b, g.choice(T, n, replace=False)] = True
    return m


def test_diagnostics_reproduce_the_references():
    g = np.random.default_rng(5)
    L, B, T, K = 16, 4, 16384, 16
    n = T // K
    ms = _repeated_masks(L, B, T, n, g)
    assert np.allclose(D.coverage(ms), 1.0 / K)
    assert np.allclose(D.adjacent_jaccard(ms), 1.0)
    cnt = D.update_counts(ms)
    assert set(np.unique(cnt)) == {0, L} and np.allclose((cnt == L).mean(axis=1), 1.0 / K)
    mr = _random_masks(L, B, T, n, g)
    cov_r, jac_r, dist_r = D.independent_random_reference(1.0 / K, L)
    assert np.all(np.abs(D.coverage(mr) - cov_r) < 4 * np.sqrt(cov_r * (1 - cov_r) / T))
    assert np.all(np.abs(D.adjacent_jaccard(mr) - jac_r) < 0.1 * jac_r)
    hist = np.bincount(D.update_counts(mr).ravel(), minlength=L + 1) / (B * T)
    assert np.abs(hist - dist_r).max() < 0.01


def _stats_from_masks(masks, logits, AK):
    """The device statistics, counted plainly: [n_sparse, B, 4] and [blocks, B, AK + 1]."""
    Ls, B, T = masks.shape
    st = np.zeros((Ls, B, 4), np.int64)
    thr = logits >= 0
    for l in range(Ls):
        st[l, :, 0] = masks[l].sum(1)
        st[l, :, 1] = thr[l].sum(1)
        st[l, :, 2] = (masks[l] == thr[l]).sum(1)
        if l % AK:
            st[l, :, 3] = np.logical_and(masks[l], masks[l - 1]).sum(1)
    blocks = Ls // AK
    uh = np.zeros((blocks, B, AK + 1), np.int64)
    for k in range(blocks):
        c = masks[k * AK:(k + 1) * AK].sum(0)
        for b in range(B):
            uh[k, b] = np.bincount(c[b], minlength=AK + 1)
    return st, uh


def test_product_diagnostics_match_the_oracle_definitions():
    g = np.random.default_rng(9)
    AK, blocks, B, T, n = 8, 2, 3, 512, 64
    masks = np.concatenate([_random_masks(AK, B, T, n, g), _repeated_masks(AK, B, T, n, g)])
    logits = g.standard_normal((blocks * AK, B, T))
    st, uh = _stats_from_masks(masks, logits, AK)
    got = PD.route_diagnostics(st, uh, T, AK)
    cov = np.mean([D.coverage(masks[k * AK:(k + 1) * AK]) for k in range(blocks)])
    jac = np.nanmean(np.concatenate([D.adjacent_jaccard(masks[k * AK:(k + 1) * AK])
                                     for k in range(blocks)]))
    assert abs(got.coverage - cov) < 1e-12
    assert abs(got.jaccard - jac) < 1e-12
    assert abs(got.agreement - D.agreement(masks, logits)) < 1e-12
    assert abs(got.threshold_rate - (logits >= 0).mean()) < 1e-12
    cnt = np.concatenate([D.update_counts(masks[k * AK:(k + 1) * AK]) for k in range(blocks)])
    assert np.allclose(got.update_dist, np.bincount(cnt.ravel(), minlength=AK + 1) / cnt.size)


def _tiny(**over):
    w = I.WORKLOADS["tiny_fp32"].replace(**over)
    layers = I.all_layer_weights(w)
    kinds = S.schedule(w.N0, w.N1, w.A, w.K)
    od = O.dims(w.B, w.T, w.d, w.hq, w.hkv, w.hd, w.F, w.eps)
    ol = [O.Layer(l) for l in layers]
    return w, kinds, od, ol, I.to_f64(I.residual_stream(w), "fp32"), I.router_bias(w)


def test_oracle_dynamics_without_growth_is_the_constant_bias_stack():
    w, kinds, od, ol, x, bias = _tiny()
    y0 = O.stack_fwd(od, w.K, w.gate, kinds, ol, x, bias=bias)
    y1, idx, s, _ = O.stack_dyn(od, w.K, w.gate, kinds, ol, x, bias=bias, bias_step=0.0)
    assert np.array_equal(y0, y1)
    assert idx.shape == (kinds.count(S.SPARSE), w.B, w.T // w.K)


def test_oracle_dynamics_overwhelming_growth_rotates_tokens():
    # [D] + ([S(4)] x 4 + [D]) x 2: blocks of K = 4 sparse layers over T = 64 tokens
    w, kinds, od, ol, x, bias = _tiny(N1=2, n_layers=1 + 2 * 5)
    big = 1e6
    y, idx, s, _ = O.stack_dyn(od, w.K, w.gate, kinds, ol, x, bias=bias, bias_step=big)
    AK, n = w.K, w.T // w.K
    masks = D.masks_from_idx(idx, w.T)
    for k in range(w.N1):
        blk = masks[k * AK:(k + 1) * AK]
        assert np.all(D.update_counts(blk) == 1)              # every token exactly once
        assert np.all(D.adjacent_jaccard(blk) == 0.0)
        assert np.all(D.coverage(blk) == 1.0)
        sb = s[k * AK:(k + 1) * AK]
        assert np.abs(sb[0]).max() < 1e3                      # cleared at the anchor
        for l in range(1, AK):
            penalised = sb[l] < -big / 2
            assert np.all(penalised.sum(axis=1) == l * n)     # earlier picks carry -big
            assert np.array_equal(penalised, blk[:l].any(axis=0))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_host_averaging_matches_plain_mask_diagnostics(seed):
    """The library's host-side averaging (sparse_depth_token_gb300.diagnostics, fed the
    per-layer and per-block counters the device gathers) against the plain mask
    diagnostics (oracle.diagnostics) on random selections and logits: coverage,
    adjacent Jaccard, agreement and the update distribution. Layers select random
    subsets of varying size (some empty, so Jaccard is undefined for some pairs), so
    the averages are not degenerate."""
    g = np.random.default_rng(seed)
    n_blocks, AK, B, T = 3, 5, 4, 40
    L = n_blocks * AK
    masks = np.zeros((L, B, T), bool)
    for l in range(L):
        for b in range(B):
            k = int(g.integers(0, 9)) if (l + b) % 7 else 0
            masks[l, b, g.choice(T, k, replace=False)] = True
    masks[AK:2 * AK, 1] = False   # one (block, sequence) with nothing selected: Jaccard undefined
    logits = g.standard_normal((L, B, T))
    # the counters of xmod_stack_fwd_ex: selected, threshold-selected, agreeing,
    # selected again after the previous sparse layer of the block
    thr = logits >= 0.0
    st = np.zeros((L, B, 4), np.int64)
    st[:, :, 0] = masks.sum(2)
    st[:, :, 1] = thr.sum(2)
    st[:, :, 2] = (masks == thr).sum(2)
    for l in range(L):
        if l % AK:
            st[l, :, 3] = np.logical_and(masks[l], masks[l - 1]).sum(1)
    uh = np.zeros((n_blocks, B, AK + 1), np.int64)
    for k in range(n_blocks):
        c = D.update_counts(masks[k * AK:(k + 1) * AK])
        for b in range(B):
            uh[k, b] = np.bincount(c[b], minlength=AK + 1)
    got = PD.route_diagnostics(st, uh, T, AK)

    cov = [D.coverage(masks[k * AK:(k + 1) * AK]) for k in range(n_blocks)]
    jac = np.concatenate([D.adjacent_jaccard(masks[k * AK:(k + 1) * AK])
                          for k in range(n_blocks)])
    assert np.isnan(jac).any() and np.isfinite(jac).sum() > 3
    np.testing.assert_allclose(got.coverage, np.mean(cov), rtol=1e-12)
    np.testing.assert_allclose(got.jaccard, np.nanmean(jac), rtol=1e-12)
    np.testing.assert_allclose(got.agreement, D.agreement(masks, logits), rtol=1e-12)
    np.testing.assert_allclose(got.threshold_rate, thr.mean(), rtol=1e-12)
    counts = np.concatenate([D.update_counts(masks[k * AK:(k + 1) * AK]).ravel()
                             for k in range(n_blocks)])
    np.testing.assert_allclose(got.update_dist, np.bincount(counts, minlength=AK + 1) / counts.size,
                               rtol=1e-12)
