"""Routing diagnostics of X-MoD notes Table 10 from the statistics that
xmod_stack_fwd_ex gathers on the device.

Inputs (host arrays, from the device tensors passed as layer_stats / update_hist):
  layer_stats [n_sparse, B, 4] int: per sparse layer (stack order) and sequence --
      selected, threshold-selected (ranked logit >= 0), agreeing decisions, and
      selected tokens the previous sparse layer of the block also selected;
  update_hist [N1, B, AK + 1] int: per sparse-dense block and sequence, tokens
      updated 0 .. AK times.
The sparse layers of block k are layer_stats[k * AK : (k + 1) * AK].

Definitions (X-MoD notes, "routing diagnostics"): coverage = share of a sequence's
tokens selected at least once in a block; adjacent-layer Jaccard = |A & B| / |A | B|
of adjacent sparse layers, averaged over the pairs with a non-empty union of each
(sequence, block) observation and then over the observations where it is defined;
mask agreement = share of token-layer positions where the top-k and threshold rules
decide alike; update counts = the distribution of how often a block updated a token.
"""
from dataclasses import dataclass

import numpy as np


@dataclass
class RouteDiagnostics:
    coverage: float            # mean over (sequence, block)
    jaccard: float             # mean over defined (sequence, block) observations
    agreement: float           # over all token-layer positions
    threshold_rate: float      # share of token-layer positions with r >= 1/2
    update_dist: np.ndarray    # [AK + 1], share of tokens updated k times in a block


def route_diagnostics(layer_stats, update_hist, T: int, AK: int) -> RouteDiagnostics:
    st = np.asarray(layer_stats, dtype=np.int64)
    uh = np.asarray(update_hist, dtype=np.int64)
    n_blocks, B, bins = uh.shape
    if bins != AK + 1 or st.shape != (n_blocks * AK, B, 4):
        raise ValueError("layer_stats / update_hist shapes do not match the stack")
    coverage = float((1.0 - uh[:, :, 0] / T).mean())
    obs = []
    for k in range(n_blocks):
        blk = st[k * AK:(k + 1) * AK]
        for b in range(B):
            vals = []
            for l in range(AK - 1):
                inter = blk[l + 1, b, 3]
                union = blk[l, b, 0] + blk[l + 1, b, 0] - inter
                if union > 0:
                    vals.append(inter / union)
            if vals:
                obs.append(np.mean(vals))
    jaccard = float(np.mean(obs)) if obs else float("nan")
    positions = st.shape[0] * B * T
    agreement = float(st[:, :, 2].sum() / positions)
    threshold_rate = float(st[:, :, 1].sum() / positions)
    update_dist = uh.sum(axis=(0, 1)) / float(n_blocks * B * T)
    return RouteDiagnostics(coverage, jaccard, agreement, threshold_rate, update_dist)
