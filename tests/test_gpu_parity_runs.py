"""Element-by-element parity of the CUDA path with the oracle over whole runs
(decode steps with periodic reassignment), through the C ABI.

Tolerances: attention outputs 2e-2 absolute (bf16 I/O, fp32 accumulate),
scores 1e-4 relative (+1e-7 absolute floor), tiers / page tables / 8-bit codes
bit-exact, values a T0/T1 token holds bit-exact.
"""
import numpy as np
import pytest
import torch

from helpers import (OUT_ATOL, assert_page_tables_equal, assert_scores_close, prefill_cache,
                     prefill_oracle)
from oracle import OracleCache
from oracle.classify import T2
from synth import CHAIN7B, MHA16K, TINY, long128k

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _run(w, steps, check_rows=True, **kw):
    from tiered_kv_cache_split_gb300 import TieredKVCache
    torch.cuda.set_device(DEV)
    cache = TieredKVCache.from_workload(w, **kw)
    oc = OracleCache.from_workload(w, t2_mode=kw.get("t2_mode", "attend"))
    prefill_cache(cache, w, DEV)
    prefill_oracle(oc, w)
    worst = 0.0
    for t in range(1, steps + 1):
        q, kn, vn = w.queries(t), w.kv_new("k", t), w.kv_new("v", t)
        out = cache.decode_step(q.to(DEV), kn.to(DEV), vn.to(DEV))
        ref, deltas = oc.decode_step(q.float().numpy(), kn.float().numpy(), vn.float().numpy())
        err = float(np.max(np.abs(out.float().cpu().numpy() - ref)))
        worst = max(worst, err)
        assert err <= OUT_ATOL, f"step {t}: output error {err}"
        for b in range(w.batch):
            assert_scores_close(cache.scores(b), oc.seqs[b].s, f"step {t} request {b}")
            assert np.array_equal(cache.tiers(b), oc.seqs[b].tier), f"step {t}: tiers of request {b}"
        if t % w.reclassify_interval == 0:
            for b in range(w.batch):
                assert_page_tables_equal(cache, oc, b, f"step {t}")
                sq = oc.seqs[b]
                for pos in np.nonzero(sq.tier == T2)[0]:
                    codes, scales = cache.t2_row(b, int(pos))
                    kc, ks, vc, vs = sq.codes[int(pos)]
                    assert np.array_equal(codes[:, 0], kc) and np.array_equal(codes[:, 1], vc), f"codes of {pos}"
                    assert np.array_equal(scales[:, 0], ks) and np.array_equal(scales[:, 1], vs), f"scales of {pos}"
                if check_rows:
                    for pos in np.nonzero(sq.tier <= 1)[0][::7]:
                        k, v = cache.kv_row(b, int(pos))
                        assert np.array_equal(k.numpy().astype(np.float64), sq.K[:, pos]), f"K row {pos}"
                        assert np.array_equal(v.numpy().astype(np.float64), sq.V[:, pos]), f"V row {pos}"
    st = cache.stats()
    assert st["steps"] == steps and st["reclassifies"] == steps // w.reclassify_interval
    cache.close()
    return worst, oc


def test_tiny_workload_whole_run():
    worst, oc = _run(TINY, TINY.n_steps)
    # tokens moved out of T2 at least once in this run (promotion path exercised)
    assert worst < 1e-4  # fp32 KV: only summation order differs


def test_tiny_workload_t2_masked_variant():
    _run(TINY, 8, t2_mode="mask")


def test_tiny_with_small_split_pages_spans_many_chunks():
    _run(TINY, 6, split_pages=8)


def test_chain7b_shape_until_all_four_tiers_exist():
    # 28 layers, 28 query / 4 KV heads, d = 128, bf16; 256-token protected prompt,
    # 128-token window, Delta = 32. Candidates appear after 128 steps, T2 after
    # ~300 and T3 after ~390: 448 steps cover 14 reassignments and every tier.
    worst, oc = _run(CHAIN7B, 448, check_rows=False)
    counts = np.bincount(oc.seqs[0].tier, minlength=4)
    assert np.all(counts > 0), counts


def test_mha_shape_with_delayed_spikes_and_per_head_fp16_scales():
    # the MHA configuration (32 query = 32 KV heads, d = 128, bf16; T2 codes with
    # one float16 scale per token and KV head; keys with delayed spikes) at 2
    # layers, 2 requests of 700 tokens and Delta = 16, so that 64 steps make four
    # reassignments over every tier.
    w = MHA16K.replace(n_layers=2, batch=2, context=("fixed", 700), prompt_len=64,
                       key_scale=("delayed_spikes", 0.02, 6.0, 40, 4), reclassify_interval=16, n_steps=64)
    worst, oc = _run(w, 64)
    for b in range(w.batch):
        assert np.all(np.bincount(oc.seqs[b].tier, minlength=4) > 0)


@pytest.mark.parametrize("t0", [25, 75])
def test_long_context_shape_without_t2(t0):
    # the long-context sweep (32 query / 8 KV heads, d = 128, bf16, lognormal(0, 1)
    # key scale, T2 = 0, T3 = 5%) at 2 layers, 2 requests of 3000 tokens, Delta = 16.
    w = long128k(t0).replace(n_layers=2, batch=2, context=("fixed", 3000), reclassify_interval=16, n_steps=48)
    worst, oc = _run(w, 48)
    for b in range(w.batch):
        counts = np.bincount(oc.seqs[b].tier, minlength=4)
        assert counts[2] == 0 and counts[0] > 0 and counts[1] > 0 and counts[3] > 0, counts


def test_reassignment_that_does_not_fit_changes_nothing():
    # Failure on the host, no GPU fault: a T1 pool of two pages cannot take the
    # tokens a reassignment sends there. The call must fail with CAPACITY and
    # leave tiers, page tables and scores as they were, and the handle usable.
    from tiered_kv_cache_split_gb300 import TieredKVCache, _lib as L
    torch.cuda.set_device(DEV)
    w = TINY
    cache = TieredKVCache.from_workload(w, t1_pages=2)
    prefill_cache(cache, w, DEV)
    cache.set_scores(0, w.synthetic_scores(0, w.context_lens()[0]).numpy())

    def snapshot():
        return cache.tiers(0).copy(), [cache.page_table(0, t) for t in range(3)], cache.scores(0).copy()

    before = snapshot()
    with pytest.raises(L.TkvError) as err:
        cache.reclassify()
    assert err.value.status == L.ERR_CAPACITY
    after = snapshot()
    assert np.array_equal(before[0], after[0]) and np.array_equal(before[2], after[2])
    for (p0, m0, q0), (p1, m1, q1) in zip(before[1], after[1]):
        assert np.array_equal(p0, p1) and np.array_equal(m0, m1) and np.array_equal(q0, q1)
    out = cache.decode_step(w.queries(1).to(DEV), w.kv_new("k", 1).to(DEV), w.kv_new("v", 1).to(DEV))
    assert bool(torch.isfinite(out.float()).all())
    cache.close()
