"""Parity at the full sizes of the MHA and long-context workloads, in the launch
configuration bench.py times.

  * MHA: 32 layers, 32 query = 32 KV heads (one query head per KV head), d = 128,
    bf16, 8 requests of 15,360 tokens with delayed key spikes; T2 in 8 bits
    with one float16 scale per token and KV head; budgets 25/50/15/10.
  * Long context: 32 layers, 32 query / 8 KV heads, d = 128, bf16, 4 requests
    of 131,072 tokens, lognormal(0, 1) key scale; budgets 50/45/0/5. Its chunk
    plan runs in three waves of ~180-page chunks.

The oracle keeps bookkeeping only (tiers, slots) and recomputes sampled
(request, layer) slices from regenerated inputs. Seeded synthetic scores put
each cache in a tiered state; then one decode step runs. Tiers, page tables
and every position's slot are compared in full, bit for bit.
"""
import numpy as np
import pytest
import torch

from helpers import (OUT_ATOL, assert_page_tables_equal, assert_scores_close, layer_attention,
                     oracle_t2_codes, prefill_cache, prefill_oracle)
from oracle import OracleCache
from synth import MHA16K, long128k

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _one_step(w):
    from tiered_kv_cache_split_gb300 import TieredKVCache
    torch.cuda.set_device(DEV)
    w = w.replace(n_steps=4)
    cache = TieredKVCache.from_workload(w)
    oc = OracleCache.from_workload(w, track_values=False)
    prefill_cache(cache, w, DEV)
    prefill_oracle(oc, w, values=False)
    s0 = []
    for b in range(w.batch):
        s = w.synthetic_scores(b, w.context_lens()[b]).numpy()
        cache.set_scores(b, s)
        oc.set_scores(b, s)
        s0.append(s)
    cache.reclassify()
    oc.reclassify()
    q = w.queries(1, DEV)
    out = cache.decode_step(q, w.kv_new("k", 1, DEV), w.kv_new("v", 1, DEV)).float().cpu().numpy()
    for b in range(w.batch):
        oc.append(b, None, None, False, n=1)
    return w, cache, oc, s0, q.float().cpu().numpy(), out


def _check_bookkeeping(w, cache, oc):
    for b in range(w.batch):
        assert np.array_equal(cache.tiers(b), oc.seqs[b].tier), f"tiers of request {b}"
        assert_page_tables_equal(cache, oc, b)


def _check_outputs(w, oc, q, out, picks):
    lens = w.context_lens()
    for b, l in picks:
        ref, _, _ = layer_attention(w, b, l, q[b, l], oc.seqs[b].tier, lens[b] + 1, gen_device=DEV)
        err = float(np.max(np.abs(out[b, l] - ref)))
        assert err <= OUT_ATOL, (b, l, err)


def _check_sum_property(w, cache, oc, s0):
    lens = w.context_lens()
    for b in range(w.batch):
        got = cache.scores(b)
        tiers = oc.seqs[b].tier
        total = (got[:lens[b]] - s0[b])[tiers[:lens[b]] != 3].sum() + got[lens[b]]
        assert abs(total - 1.0) < 1e-4, (b, total)


def test_mha_workload_at_full_size():
    w, cache, oc, s0, q, out = _one_step(MHA16K)
    try:
        _check_bookkeeping(w, cache, oc)
        counts = np.bincount(np.concatenate([oc.seqs[b].tier for b in range(w.batch)]), minlength=4)
        assert np.all(counts > 0), counts
        _check_outputs(w, oc, q, out, [(0, 0), (3, 17), (7, 31), (5, 8)])
        _check_sum_property(w, cache, oc, s0)
        # every layer's weights of one request, position by position
        b, n_total = 6, w.context_lens()[6] + 1
        acc = np.zeros(n_total)
        for l in range(w.n_layers):
            _, alpha, R = layer_attention(w, b, l, q[b, l], oc.seqs[b].tier, n_total, gen_device=DEV)
            acc[R] += alpha.mean(axis=0)
        assert_scores_close(cache.scores(b), np.concatenate([s0[b], [0.0]]) + acc / w.n_layers, f"request {b}")
        rng = np.random.default_rng(3)
        for b in (1, 4):
            pos2 = np.nonzero(oc.seqs[b].tier == 2)[0]
            for pos in rng.choice(pos2, size=3, replace=False):
                codes, scales = cache.t2_row(b, int(pos))
                (kc, ks), (vc, vs) = oracle_t2_codes(w, b, int(pos))
                assert np.array_equal(codes[:, 0], kc) and np.array_equal(codes[:, 1], vc)
                assert np.array_equal(scales[:, 0], ks) and np.array_equal(scales[:, 1], vs)
    finally:
        cache.close()
        del cache
        torch.cuda.empty_cache()


def test_long_context_workload_at_full_size():
    w, cache, oc, s0, q, out = _one_step(long128k(50))
    try:
        _check_bookkeeping(w, cache, oc)
        counts = np.bincount(np.concatenate([oc.seqs[b].tier for b in range(w.batch)]), minlength=4)
        assert counts[2] == 0 and counts[0] > 0 and counts[1] > 0 and counts[3] > 0, counts
        _check_outputs(w, oc, q, out, [(0, 0), (1, 31), (2, 16), (3, 5)])
        _check_sum_property(w, cache, oc, s0)
    finally:
        cache.close()
        del cache
        torch.cuda.empty_cache()
