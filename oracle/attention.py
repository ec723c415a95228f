"""Decode attention over the retained set, in float64.

Methodology 3 ("Not All Thoughts Need HBM", zero-approximation-error offload):
a T1 token is prefetched at full precision before attention, so it contributes
exactly the term it would have contributed from HBM; attention therefore runs
over every retained token (T0, T1 and T2, with T2 dequantised), and only the
evicted set T3 is absent.

The attention itself is the textbook single-query softmax attention of one
decode step with grouped query heads (query head h reads key/value head
h // (Hq / Hkv)); the softmax scale 1/sqrt(d) is the standard one (the pages do
not state it). Pins: a hand-worked 3-token case, brute-force agreement with
torch's float64 scaled_dot_product_attention when nothing is evicted, and a
GQA test where each KV head holds distinct values.
"""
from __future__ import annotations

import math

import numpy as np


def decode_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray):
    """One decode step of attention for one request at one layer.

    q: [Hq, d] query of the new token; K, V: [n, Hkv, d] the retained keys and
    values (float64, in the precision each tier holds). Returns
    (out [Hq, d], alpha [Hq, n]) where alpha[h] is head h's softmax weights.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    Hq, d = q.shape
    n, Hkv, _ = K.shape
    if n == 0:
        raise ValueError("decode attention over an empty retained set")
    G = Hq // Hkv
    out = np.empty((Hq, d), dtype=np.float64)
    alpha = np.empty((Hq, n), dtype=np.float64)
    for h in range(Hq):
        kvh = h // G
        logits = (K[:, kvh, :] @ q[h]) / math.sqrt(d)
        e = np.exp(logits - logits.max())
        a = e / e.sum()
        alpha[h] = a
        out[h] = a @ V[:, kvh, :]
    return out, alpha
