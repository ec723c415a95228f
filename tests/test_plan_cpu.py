"""The attention work plan of a decode step, checked on the CPU through the
library's host-only hook (tkv_test_plan_attention): how each sequence's page
list is split into chunks, and the order in which the launch hands its units
out. No device is involved.

Invariants:
  * every sequence gets 1..128 chunks; no chunk costs more than a CTA may take
    (255 full-page units of cost, so at most 256 pages), and the returned page
    bound covers the largest chunk;
  * automatic splitting keeps at least ~8 pages per chunk, and adds chunks only
    up to whole waves of resident CTAs (at most 8 waves);
  * a fixed split_pages gives each sequence ceil(pages / split_pages) chunks,
    within the same limits;
  * the hand-out order is a permutation of the sequences by decreasing chunk
    cost, ties by index, and its prefix sums match the chunk counts.
"""
import ctypes
import math

import numpy as np
import pytest

from tiered_kv_cache_split_gb300 import _lib as L

COST_FULL, COST_I8, MAX_CHUNK_PAGES, MAX_CHUNKS = 2, 3, 256, 128
MAX_CHUNK_COST = COST_FULL * (MAX_CHUNK_PAGES - 1)


@pytest.fixture(scope="module")
def lib():
    import os
    if not os.path.exists(L.LIB_PATH):
        from tiered_kv_cache_split_gb300 import build
        build.build()
    return L.load()


def _plan(lib, full, i8, hkv, split, resident):
    B = len(full)
    full = np.ascontiguousarray(full, dtype=np.int64)
    i8 = np.ascontiguousarray(i8, dtype=np.int64)
    chunk_first = np.zeros(B + 1, dtype=np.int32)
    order = np.zeros(B, dtype=np.int32)
    ocf = np.zeros(B + 1, dtype=np.int32)
    bound = ctypes.c_int32()
    st = lib.tkv_test_plan_attention(B, full.ctypes.data, i8.ctypes.data, hkv, split, resident,
                                     chunk_first.ctypes.data, order.ctypes.data, ocf.ctypes.data,
                                     ctypes.byref(bound))
    L.check(st)
    return chunk_first, order, ocf, bound.value


def _check(full, i8, hkv, split, resident, chunk_first, order, ocf, bound):
    B = len(full)
    nch = np.diff(chunk_first)
    ntot = np.asarray(full) + np.asarray(i8)
    cost = COST_FULL * np.asarray(full) + COST_I8 * np.asarray(i8)
    assert chunk_first[0] == 0 and np.all(nch >= 1) and np.all(nch <= MAX_CHUNKS), nch
    for b in range(B):
        floor_b = max(1, math.ceil(cost[b] / MAX_CHUNK_COST))
        assert cost[b] <= nch[b] * MAX_CHUNK_COST, (b, cost[b], nch[b])          # a chunk fits one CTA
        assert nch[b] >= floor_b
        if split == 0:
            assert nch[b] <= max(floor_b, min(MAX_CHUNKS, max(1, math.ceil(ntot[b] / 8)))), (b, nch[b])
        else:
            want = max(floor_b, math.ceil(max(ntot[b], 1) / split))
            assert nch[b] == min(max(floor_b, min(MAX_CHUNKS, max(1, math.ceil(ntot[b] / 8)))), want), (b, nch[b])
        # the largest chunk of b holds at most ceil(cost / nch) cost units + one page of rounding
        assert bound >= min(ntot[b], math.ceil(cost[b] / (nch[b] * COST_FULL)))
    assert bound <= MAX_CHUNK_PAGES
    if split == 0:
        waves = min(8, max(1, math.ceil(ntot.sum() * hkv / (resident * 240))))
        target = max(B, waves * resident // hkv)
        floors = sum(max(1, math.ceil(c / MAX_CHUNK_COST)) for c in cost)
        assert nch.sum() <= max(target, floors), (nch.sum(), target, floors)
    # hand-out order: a permutation, chunk cost non-increasing, ties by index
    assert sorted(order.tolist()) == list(range(B))
    for r in range(B - 1):
        x, y = order[r], order[r + 1]
        lhs, rhs = int(cost[x]) * int(nch[y]), int(cost[y]) * int(nch[x])
        assert lhs > rhs or (lhs == rhs and x < y), (r, x, y)
    assert ocf[0] == 0 and np.array_equal(np.diff(ocf), nch[order])


@pytest.mark.parametrize("seed", range(12))
def test_random_plans_keep_their_invariants(lib, seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 65))
    kind = seed % 4
    if kind == 0:      # the batch-32 mix: uniform lengths, a T2 share
        full = rng.integers(50, 460, size=B)
        i8 = rng.integers(0, 60, size=B)
    elif kind == 1:    # long contexts near the page limit
        full = rng.integers(4000, 15000, size=B)
        i8 = rng.integers(0, 1300, size=B)
    elif kind == 2:    # tiny and empty lists
        full = rng.integers(0, 5, size=B)
        i8 = rng.integers(0, 3, size=B)
    else:              # a heavy tail
        full = np.minimum(16000, (rng.pareto(1.2, size=B) * 200).astype(np.int64) + 1)
        i8 = np.zeros(B, dtype=np.int64)
    hkv = int(rng.choice([1, 2, 4, 8, 32]))
    resident = int(rng.choice([152, 304, 456]))
    split = 0 if seed % 3 else int(rng.choice([8, 32, 80]))
    res = _plan(lib, full, i8, hkv, split, resident)
    _check(full.tolist(), i8.tolist(), hkv, split, resident, *res)


def test_the_batch32_shape_fills_one_wave_largest_chunks_first(lib):
    # 32 sequences of 1k..8k tokens at 40/40/10/10: ~10k pages, 4 KV heads, 456 resident CTAs
    rng = np.random.default_rng(13)
    tokens = rng.integers(1024, 8193, size=32)
    full = (tokens * 0.8 / 16).astype(np.int64) + 1
    i8 = (tokens * 0.1 / 16).astype(np.int64) + 1
    chunk_first, order, ocf, bound = _plan(lib, full, i8, 4, 0, 456)
    _check(full.tolist(), i8.tolist(), 4, 0, 456, chunk_first, order, ocf, bound)
    assert chunk_first[-1] * 4 == 456            # exactly one wave of units per layer
    nch = np.diff(chunk_first)
    cost = COST_FULL * full + COST_I8 * i8
    per_chunk = cost[order] / nch[order]
    assert per_chunk[0] == per_chunk.max() and per_chunk[-1] == per_chunk.min()


def test_bad_arguments_are_refused(lib):
    one = np.ones(1, dtype=np.int64)
    out = np.zeros(2, dtype=np.int32)
    b = ctypes.c_int32()
    args = lambda n, full, h, s, r: lib.tkv_test_plan_attention(n, full.ctypes.data, one.ctypes.data, h, s, r,
                                                                out.ctypes.data, out.ctypes.data, out.ctypes.data,
                                                                ctypes.byref(b))
    assert args(0, one, 4, 0, 456) == L.ERR_INVALID_ARG
    assert args(65, one, 4, 0, 456) == L.ERR_INVALID_ARG
    assert args(1, np.array([-1], dtype=np.int64), 4, 0, 456) == L.ERR_INVALID_ARG
    assert args(1, np.array([16384], dtype=np.int64), 4, 0, 456) == L.ERR_INVALID_ARG   # with the T2 page: 16385
    assert args(1, one, 0, 0, 456) == L.ERR_INVALID_ARG
    assert args(1, one, 4, -1, 456) == L.ERR_INVALID_ARG
    assert args(1, one, 4, 0, 0) == L.ERR_INVALID_ARG
    assert args(1, one, 4, 0, 456) == L.OK
