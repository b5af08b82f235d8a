"""Routing diagnostics of a sparse-dense block, computed plainly from selection masks.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py): the CUDA library never imports this.

Definitions follow "X-MoD: Practical Scaling Laws for Sparse-Depth Routing Beyond
Mixture-of-Depths" (reading notes), section "routing diagnostics" and Table 10:
  coverage   fraction of a sequence's tokens selected at least once over the run of
             consecutive sparse layers between dense anchors;
  Jaccard    overlap of the token sets of adjacent sparse layers, averaged over the
             layer pairs with a non-empty union inside each (sequence, run)
             observation, then over the observations where it is defined;
  agreement  fraction of token-layer positions where the top-k mask and the causal
             threshold mask (routing probability >= 1/2, i.e. logit >= 0) computed on
             the same logits make the same binary decision;
  updates    how many of the run's layers updated each token.
And the two analytic references of that section, with nominal rate p = 1/K over a
run of L layers: the same subset every layer (coverage p, Jaccard 1, updates 0 with
probability 1 - p and L with probability p) and independent random subsets (coverage
1 - (1 - p)^L, Jaccard about p / (2 - p), updates Binomial(L, p))."""
from math import comb

import numpy as np


def masks_from_idx(idx, T):
    """idx [L, B, n] selected positions -> boolean masks [L, B, T]."""
    idx = np.asarray(idx)
    L, B, _ = idx.shape
    m = np.zeros((L, B, T), bool)
    for l in range(L):
        for b in range(B):
            m[l, b, idx[l, b]] = True
    return m


def coverage(masks):
    """masks [L, B, T] of one run -> per-sequence coverage [B]."""
    return np.asarray(masks).any(axis=0).mean(axis=1)


def adjacent_jaccard(masks):
    """masks [L, B, T] of one run -> per-sequence mean adjacent-layer Jaccard [B]
    (NaN where no adjacent pair has a non-empty union)."""
    m = np.asarray(masks)
    L, B, _ = m.shape
    out = np.full(B, np.nan)
    for b in range(B):
        vals = []
        for l in range(L - 1):
            inter = np.logical_and(m[l, b], m[l + 1, b]).sum()
            union = np.logical_or(m[l, b], m[l + 1, b]).sum()
            if union > 0:
                vals.append(inter / union)
        if vals:
            out[b] = float(np.mean(vals))
    return out


def update_counts(masks):
    """masks [L, B, T] -> how many layers selected each token [B, T]."""
    return np.asarray(masks).sum(axis=0)


def agreement(topk_masks, logits):
    """Fraction of positions where the top-k mask equals the threshold mask logit >= 0."""
    thr = np.asarray(logits) >= 0.0
    return float((np.asarray(topk_masks) == thr).mean())


def repeated_subset_reference(p, L):
    """(coverage, Jaccard, update-count distribution over 0..L) of the same subset."""
    dist = np.zeros(L + 1)
    dist[0], dist[L] = 1.0 - p, p
    return p, 1.0, dist


def independent_random_reference(p, L):
    """(coverage, Jaccard, update-count distribution) of independent random subsets."""
    dist = np.array([comb(L, k) * p**k * (1.0 - p) ** (L - k) for k in range(L + 1)])
    return 1.0 - (1.0 - p) ** L, p / (2.0 - p), dist
