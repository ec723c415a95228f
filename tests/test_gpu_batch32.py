"""Parity at the full batch-32 serving size (the benchmarked workload), in the
launch configuration bench.py times: 32 requests of 1k-8k tokens, 28 layers,
28 query / 4 KV heads, d = 128, bf16, budgets 40/40/10/10.

The oracle cannot hold 8.5 GB of float64 state at once, so it keeps
bookkeeping only (tiers, slots) and recomputes, one (request, layer) at a time
from regenerated inputs, every request's scores and all layers and heads of
four requests' outputs. Seeded synthetic scores put the cache in a tiered
state; then one decode step runs.
"""
import numpy as np
import pytest
import torch

from helpers import (OUT_ATOL, assert_page_tables_equal, assert_scores_close, layer_attention,
                     oracle_t2_codes, prefill_cache, prefill_oracle)
from oracle import OracleCache
from synth import BATCH32

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def state():
    from tiered_kv_cache_split_gb300 import TieredKVCache
    torch.cuda.set_device(DEV)
    w = BATCH32
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
    tiers_before = [oc.seqs[b].tier.copy() for b in range(w.batch)]
    q, kn, vn = w.queries(1), w.kv_new("k", 1), w.kv_new("v", 1)
    out = cache.decode_step(q.to(DEV), kn.to(DEV), vn.to(DEV)).float().cpu().numpy()
    for b in range(w.batch):
        oc.append(b, None, None, False, n=1)
    yield dict(w=w, cache=cache, oc=oc, s0=s0, q=q.float().numpy(), out=out, tiers=tiers_before)
    cache.close()
    del cache
    torch.cuda.empty_cache()


def test_tiers_and_page_tables_bit_exact(state):
    cache, oc, w = state["cache"], state["oc"], state["w"]
    for b in range(w.batch):
        assert np.array_equal(cache.tiers(b), oc.seqs[b].tier), f"tiers of request {b}"
        assert_page_tables_equal(cache, oc, b)
    counts = np.bincount(np.concatenate([oc.seqs[b].tier for b in range(w.batch)]), minlength=4)
    assert np.all(counts > 0)


@pytest.fixture(scope="module")
def oracle_pass(state):
    """The oracle over every (request, layer) of the step: all heads' outputs of
    four requests (the shortest, two of median length, the longest), and every
    request's score increments. Inputs are regenerated on the device (the same
    bits as on the CPU) and all arithmetic runs in float64 on the CPU."""
    w, q = state["w"], state["q"]
    lens = w.context_lens()
    order = [int(i) for i in np.argsort(lens)]
    picked = {order[0], order[15], order[16], order[-1]}
    outs, scores = {}, {}
    for b in range(w.batch):
        n_total = lens[b] + 1
        tiers = state["oc"].seqs[b].tier
        acc = np.zeros(n_total)
        for l in range(w.n_layers):
            ref, alpha, R = layer_attention(w, b, l, q[b, l], tiers, n_total, gen_device=DEV)
            acc[R] += alpha.mean(axis=0)
            if b in picked:
                outs[(b, l)] = ref
        scores[b] = np.concatenate([state["s0"][b], [0.0]]) + acc / w.n_layers
    return outs, scores


def test_outputs_of_four_requests_every_layer_and_head(state, oracle_pass):
    outs, _ = oracle_pass
    worst = 0.0
    for (b, l), ref in outs.items():
        err = float(np.max(np.abs(state["out"][b, l] - ref)))
        worst = max(worst, err)
        assert err <= OUT_ATOL, (b, l, err)
    assert len(outs) == 4 * state["w"].n_layers


def test_scores_of_every_request_and_sum_property(state, oracle_pass):
    w, cache, oc = state["w"], state["cache"], state["oc"]
    _, want = oracle_pass
    lens = w.context_lens()
    for b in range(w.batch):
        got = cache.scores(b)
        ds = got[:lens[b]] - state["s0"][b]
        tiers = oc.seqs[b].tier
        # one step: increments over the retained set sum to 1 (the new token's
        # own weight is its score, since its previous score is 0)
        total = ds[tiers[:lens[b]] != 3].sum() + got[lens[b]]
        assert abs(total - 1.0) < 1e-4, (b, total)
        assert_scores_close(got, want[b], f"request {b}")


def test_sampled_t2_codes(state):
    w, cache, oc = state["w"], state["cache"], state["oc"]
    rng = np.random.default_rng(0)
    for b in (0, 7, 31):
        pos2 = np.nonzero(oc.seqs[b].tier == 2)[0]
        for pos in rng.choice(pos2, size=min(4, len(pos2)), replace=False):
            codes, scales = cache.t2_row(b, int(pos))
            (kc, ks), (vc, vs) = oracle_t2_codes(w, b, int(pos))
            assert np.array_equal(codes[:, 0], kc) and np.array_equal(codes[:, 1], vc)
            assert np.array_equal(scales[:, 0], ks) and np.array_equal(scales[:, 1], vs)
