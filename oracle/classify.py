"""Tier reassignment, step by step, in plain Python.

Methodology 1 ("Not All Thoughts Need HBM", four-tier classification): T0 (HBM)
holds the protected tokens — the prompt, the attention sinks and the recent
window — plus the most important reasoning tokens; T1 (DDR, full precision)
the medium ones; T2 (8-bit) the low ones; T3 only the absolute tail, deleted
for good. Methodology 4: the assignment is recomputed every Delta decode steps.

Readings where the page is silent (each the plainest one):
  * the protected set is [0, max(prompt_len, n_sink)) together with the last
    W positions [N - W, N);
  * budgets are integer fractions of the N positions seen so far:
    n1 = floor(p1 N / 100), n2 = floor(p2 N / 100), n3 = floor(p3 N / 100),
    n0 = N - n1 - n2 - n3 (or absolute counts n0, n1, n2 with T3 the rest);
  * candidates are the positions neither protected nor already evicted; they
    are ranked by score descending, ties by lower position first (-0 equals
    +0); the first max(n0 - |P|, 0) go to T0, the next n1 to T1, the next n2
    to T2 and the rest to T3, taking fewer where candidates run out;
  * eviction is permanent: an already-T3 position stays T3.
Pins: brute-force enumeration of every assignment with the right counts on
n <= 8 positions, hand-worked fixtures, and the ordering invariants.
"""
from __future__ import annotations

import numpy as np

T0, T1, T2, T3 = 0, 1, 2, 3


def protected_mask(N: int, prompt_len: int, n_sink: int, recent_window: int) -> np.ndarray:
    P = np.zeros(N, dtype=bool)
    P[:min(N, max(prompt_len, n_sink))] = True
    P[max(N - recent_window, 0):] = True
    return P


def budgets_for(N: int, mode: str, budgets) -> tuple[int, int, int]:
    """(n0, n1, n2) for N positions."""
    if mode == "count":
        return int(budgets[0]), int(budgets[1]), int(budgets[2])
    n1 = budgets[1] * N // 100
    n2 = budgets[2] * N // 100
    n3 = budgets[3] * N // 100
    return N - n1 - n2 - n3, n1, n2


def classify(s, old_tier, prompt_len: int, n_sink: int, recent_window: int,
             n0: int, n1: int, n2: int) -> np.ndarray:
    """New tier (uint8 [N]) of every position of one request."""
    s = [float(x) for x in s]
    old = np.asarray(old_tier, dtype=np.uint8)
    N = len(s)
    P = protected_mask(N, prompt_len, n_sink, recent_window)
    if np.any(P & (old == T3)):
        raise ValueError("a protected position is already evicted")
    new = old.copy()
    new[P] = T0
    candidates = [i for i in range(N) if not P[i] and old[i] != T3]
    # score descending, then position ascending; 0.0 == -0.0 in this comparison
    ranked = sorted(candidates, key=lambda i: (-s[i], i))
    a0 = max(n0 - int(P.sum()), 0)
    for rank, i in enumerate(ranked):
        if rank < a0:
            new[i] = T0
        elif rank < a0 + n1:
            new[i] = T1
        elif rank < a0 + n1 + n2:
            new[i] = T2
        else:
            new[i] = T3
    return new
