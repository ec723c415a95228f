"""Cumulative attention score increment, in float64.

Methodology 2 ("Not All Thoughts Need HBM", importance scoring): at decode step
t the score of position i grows by the attention weight it received, averaged
over the heads of each layer and then over the layers:

    s_i(t) = s_i(t-1) + (1/|L|) * sum over layers l of (1/H) * sum over heads h
             of alpha_{l,h}(t)[i]

Reading: H is the number of query heads (alpha is per query head) and L is
every layer. Pins: the increments of one step sum to 1 over the retained set,
and with one layer and one head the increment is that head's attention row.
"""
from __future__ import annotations

import numpy as np


def score_increment(alphas) -> np.ndarray:
    """alphas: per layer, an [H, n] array of softmax weights over the same n
    retained positions. Returns the [n] increment of s for this step."""
    L = len(alphas)
    total = None
    for a in alphas:
        a = np.asarray(a, dtype=np.float64)
        H = a.shape[0]
        layer_mean = a.sum(axis=0) / H
        total = layer_mean if total is None else total + layer_mean
    return total / L
