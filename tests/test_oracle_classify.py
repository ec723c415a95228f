"""Pins of the oracle's tier reassignment (CPU only).

"Not All Thoughts Need HBM", Methodology 1 (four tiers; protected prompt,
sinks and recent window in T0; only the tail evicted) and Methodology 4
(periodic reassignment).
"""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import budgets_for, classify, protected_mask
from oracle.classify import T0, T1, T2, T3


def test_hand_worked_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "classify_example.json")))
    new = classify(g["scores"], g["old_tier"], g["prompt_len"], g["n_sink"],
                   g["recent_window"], g["n0"], g["n1"], g["n2"])
    assert new.tolist() == g["new_tier"]


def _brute_force(s, old, P, n0, n1, n2):
    """The unique assignment of the candidates, with the truncated counts, in
    which every token of a better tier beats every token of a worse tier by
    (score desc, position asc) — found by enumerating all assignments."""
    N = len(s)
    cand = [i for i in range(N) if not P[i] and old[i] != T3]
    c = len(cand)
    a0 = max(n0 - int(P.sum()), 0)
    k0 = min(a0, c)
    k1 = min(n1, c - k0)
    k2 = min(n2, c - k0 - k1)
    k3 = c - k0 - k1 - k2
    labels = [T0] * k0 + [T1] * k1 + [T2] * k2 + [T3] * k3
    found = []
    for perm in set(itertools.permutations(labels)):
        ok = True
        for x, i in enumerate(cand):
            for y, j in enumerate(cand):
                if perm[x] < perm[y]:
                    beats = s[i] > s[j] or (s[i] == s[j] and i < j)
                    if not beats:
                        ok = False
                        break
            if not ok:
                break
        if ok:
            found.append(perm)
    assert len(found) == 1
    new = np.array(old, dtype=np.uint8)
    new[P] = T0
    for x, i in enumerate(cand):
        new[i] = found[0][x]
    return new


@pytest.mark.parametrize("seed", range(40))
def test_brute_force_small(seed):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(1, 9))
    s = rng.integers(0, 4, N) / 4.0            # many ties
    if seed % 5 == 0:
        s = -s * 0.0                           # -0.0 and +0.0 must tie
    prompt, sink, W = int(rng.integers(0, 3)), int(rng.integers(0, 2)), int(rng.integers(0, 3))
    P = protected_mask(N, prompt, sink, W)
    old = np.zeros(N, dtype=np.uint8)
    for i in range(N):
        if not P[i] and rng.random() < 0.25:
            old[i] = T3
        elif not P[i]:
            old[i] = rng.integers(0, 3)
    n0, n1, n2 = (int(x) for x in rng.integers(0, 4, 3))
    new = classify(s, old, prompt, sink, W, n0, n1, n2)
    assert new.tolist() == _brute_force(s, old, P, n0, n1, n2).tolist()


def test_invariants_on_a_large_random_case():
    rng = np.random.default_rng(1)
    N = 3000
    s = np.floor(rng.random(N) * 50) / 50
    old = np.zeros(N, dtype=np.uint8)
    old[rng.choice(np.arange(300, 2800), 150, replace=False)] = T3
    n0, n1, n2 = budgets_for(N, "percent", (40, 40, 10, 10))
    new = classify(s, old, 256, 4, 128, n0, n1, n2)
    P = protected_mask(N, 256, 4, 128)
    assert np.all(new[P] == T0)
    assert np.all(new[old == T3] == T3)                       # eviction is permanent
    counts = np.bincount(new, minlength=4)
    assert counts[1] == n1 and counts[2] == n2 and counts[0] == n0
    cand = ~P & (old != T3)
    for a, b in ((T0, T1), (T1, T2), (T2, T3)):
        worse = cand & (new == b) if b != T3 else cand & (new == T3)
        better = cand & (new == a)
        if better.any() and worse.any():
            assert s[better].min() >= s[worse].max()


def test_budgets_percent_and_count():
    assert budgets_for(1000, "percent", (40, 40, 10, 10)) == (400, 400, 100)
    assert budgets_for(1029, "percent", (40, 40, 10, 10)) == (1029 - 411 - 102 - 102, 411, 102)
    assert budgets_for(512, "count", (256, 128, 64, 0)) == (256, 128, 64)


def test_protected_larger_than_t0_budget_takes_from_t3_first():
    N = 10
    s = np.arange(N, dtype=np.float64)
    old = np.zeros(N, dtype=np.uint8)
    # protected {0..5} (6 tokens) > n0 = 4: no candidate goes to T0, T1/T2 are
    # filled and only the rest is evicted.
    new = classify(s, old, 6, 0, 0, 4, 2, 1)
    assert new.tolist() == [0, 0, 0, 0, 0, 0, 3, 2, 1, 1]


def test_protected_sets_by_hand(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "protected_sets.json")))
    for c in g["cases"]:
        P = protected_mask(c["N"], c["prompt_len"], c["n_sink"], c["recent_window"])
        assert np.nonzero(P)[0].tolist() == c["protected"], c["name"]
    x = g["classify_with_sinks_beyond_prompt"]
    new = classify(x["scores"], x["old_tier"], x["prompt_len"], x["n_sink"], x["recent_window"],
                   x["n0"], x["n1"], x["n2"])
    assert new.tolist() == x["new_tier"]
