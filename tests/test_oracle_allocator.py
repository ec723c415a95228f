"""Pins of the oracle's slot allocator (CPU only).

"Not All Thoughts Need HBM", Methodology 4: only tokens whose tier changed
move; the reading fixes where they land (ascending holes, then new pages).
"""
import json
import os

import numpy as np

from oracle import PagedAllocator


def test_hand_worked_two_pages(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "allocator_2page.json")))
    a = PagedAllocator(16)
    for op, b, pos in g["ops"]:
        getattr(a, op)(b, pos)
    for b, table in g["tables"].items():
        assert [[p, s] for p, s in a.table(int(b))] == table


def test_hand_worked_compaction_and_page_reuse(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "allocator_compact.json")))
    a = PagedAllocator(16)
    moves = None
    for op, b, pos in g["ops"]:
        if op == "compact":
            moves = a.compact(b)
        else:
            getattr(a, op)(b, pos)
    assert [[m[0], list(m[1]), list(m[2])] for m in moves] == g["moves"]
    for b, table in g["tables"].items():
        assert [[p, s] for p, s in a.table(int(b))] == table
    assert a.next_page == g["next_page"]


def test_random_operations_keep_invariants():
    rng = np.random.default_rng(0)
    a = PagedAllocator(16)
    held = {0: set(), 1: set(), 2: set()}
    nxt = {0: 0, 1: 0, 2: 0}
    for _ in range(300):
        b = int(rng.integers(0, 3))
        if held[b] and rng.random() < 0.1:
            a.compact(b)
            n = len(held[b])
            assert len(a.pages[b]) == -(-n // 16)
        elif held[b] and rng.random() < 0.4:
            out = rng.choice(sorted(held[b]), size=min(len(held[b]), int(rng.integers(1, 9))), replace=False)
            a.vacate(b, out)
            held[b] -= set(int(x) for x in out)
        else:
            k = int(rng.integers(1, 20))
            new = list(range(nxt[b], nxt[b] + k))
            nxt[b] += k
            a.place(b, new)
            held[b] |= set(new)
    seen_pages = set()
    for b in range(3):
        table = a.table(b)
        ids = [p for p, _ in table]
        assert ids == sorted(ids) and not (set(ids) & seen_pages)
        seen_pages |= set(ids)
        occupied = [x for _, slots in table for x in slots if x >= 0]
        assert sorted(occupied) == sorted(held[b])                  # popcount == count
        assert len(occupied) == len(set(occupied))                  # no double booking
    assert seen_pages | set(a.free) == set(range(a.next_page))
    assert not (seen_pages & set(a.free))
