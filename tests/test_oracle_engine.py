"""Pins of the oracle's whole step loop (CPU only).

"Not All Thoughts Need HBM": Methodology 1 (tiers and budgets), 2 (scores),
3 (Proposition 1: the error depends only on T3, not on the T0/T1 split) and 4
(reassignment every Delta steps).
"""
import numpy as np
import pytest

from oracle import OracleCache
from oracle.classify import T0, T1, T2, T3, protected_mask
from synth import TINY


def _run_tiny(steps=None, **kw):
    w = TINY
    oc = OracleCache.from_workload(w, **kw)
    n = w.context_lens()[0]
    oc.append(0, w.kv_layers("k", 0, 0, w.prompt_len).numpy(),
              w.kv_layers("v", 0, 0, w.prompt_len).numpy(), True)
    oc.append(0, w.kv_layers("k", 0, w.prompt_len, n).numpy(),
              w.kv_layers("v", 0, w.prompt_len, n).numpy(), False)
    outs = []
    for t in range(1, (steps or w.n_steps) + 1):
        out, deltas = oc.decode_step(w.queries(t).numpy(), w.kv_new("k", t).numpy(),
                                     w.kv_new("v", t).numpy())
        outs.append((out, deltas, oc.seqs[0].tier.copy()))
    return oc, outs


def test_tiny_run_invariants():
    oc, outs = _run_tiny()
    w = TINY
    prev_t3 = np.zeros(0, dtype=bool)
    for t, (out, deltas, tier) in enumerate(outs, start=1):
        R, ds = deltas[0]
        assert abs(ds.sum() - 1.0) < 1e-12                       # sum of increments is 1
        assert np.all(ds >= 0)
        N = len(tier)
        P = protected_mask(N, w.prompt_len, w.n_sink, w.recent_window)
        assert np.all(tier[P] == T0)
        t3 = tier == T3
        assert np.all(t3[:len(prev_t3)] >= prev_t3)              # eviction is permanent
        prev_t3 = t3
        if t % w.reclassify_interval == 0:
            c = np.bincount(tier, minlength=4)
            assert (c[0], c[1], c[2]) == (256, 128, 64) and c[3] == N - 448
    sq = oc.seqs[0]
    # page tables hold exactly the tokens of each tier
    for x in (T0, T1, T2):
        held = [p for _, slots in oc.page_table(0, x) for p in slots if p >= 0]
        assert sorted(held) == np.nonzero(sq.tier == x)[0].tolist()
    assert set(sq.codes) == set(np.nonzero(sq.tier == T2)[0].tolist())


def test_proposition_1_t1_split_changes_nothing():
    # Two caches with identical contents; one reassigns half of the
    # unprotected tokens to T1 (no T2, no T3), the other keeps all in T0.
    w = TINY
    a = OracleCache.from_workload(w, )
    b = OracleCache.from_workload(w)
    a.budget_mode = "count"; a.budgets = (200, 600, 0, 0)
    b.budget_mode = "count"; b.budgets = (800, 0, 0, 0)
    n = w.context_lens()[0]
    for oc in (a, b):
        oc.append(0, w.kv_layers("k", 0, 0, 32).numpy(), w.kv_layers("v", 0, 0, 32).numpy(), True)
        oc.append(0, w.kv_layers("k", 0, 32, n).numpy(), w.kv_layers("v", 0, 32, n).numpy(), False)
        oc.set_scores(0, w.synthetic_scores(0, n).numpy())
        oc.reclassify()
    assert np.count_nonzero(a.seqs[0].tier == T1) > 200
    assert np.all(b.seqs[0].tier == T0)
    for t in range(1, 4):
        args = (w.queries(t).numpy(), w.kv_new("k", t).numpy(), w.kv_new("v", t).numpy())
        oa, da = a.decode_step(*args)
        ob, db = b.decode_step(*args)
        assert np.max(np.abs(oa - ob)) <= 1e-12
        np.testing.assert_allclose(da[0][1], db[0][1], rtol=0, atol=1e-12)


def test_t2_tokens_are_read_dequantised_and_t3_absent():
    oc, outs = _run_tiny(steps=4)
    sq = oc.seqs[0]
    pos2 = np.nonzero(sq.tier == T2)[0]
    assert len(pos2) == 64
    kc, ks, vc, vs = sq.codes[int(pos2[0])]
    np.testing.assert_array_equal(sq.K[:, pos2[0]], kc.astype(np.float64) * np.float64(ks[0]))
    R = oc.retained(0)
    assert not np.any(sq.tier[R] == T3) and len(R) == sq.N - np.count_nonzero(sq.tier == T3)


def test_kv_size_of_a_2000_token_chain_is_about_800_mb():
    # Problem statement: a 2,000-token chain on a 7B model holds ~800 MB of KV.
    # 28 layers x 28 KV heads x 128 dims x (K, V) x 2 bytes x 2,000 tokens:
    assert 2000 * 28 * 28 * 128 * 2 * 2 == 802_816_000


def test_one_layer_two_steps_by_hand(golden_dir):
    """The new token is appended before attention (its own query sees it) and
    scores accumulate the head- and layer-averaged weights across steps."""
    import json
    import os
    g = json.load(open(os.path.join(golden_dir, "decode_step_1layer.json")))
    oc = OracleCache(g["n_layers"], g["n_q_heads"], g["n_kv_heads"], g["head_dim"], "f32", n_sink=0,
                     recent_window=0, budget_mode="count", budgets=(100, 0, 0, 0), reclassify_interval=1000)
    k = np.array(g["prompt_k"], dtype=np.float64)[None]     # [L, n, Hkv, d]
    v = np.array(g["prompt_v"], dtype=np.float64)[None]
    oc.append(0, k, v, True)
    for st in g["steps"]:
        q = np.array(st["q"], dtype=np.float64)[None, None]           # [B, L, Hq, d]
        kn = np.array(st["k_new"], dtype=np.float64)[None, None]      # [B, L, Hkv, d]
        vn = np.array(st["v_new"], dtype=np.float64)[None, None]
        out, deltas = oc.decode_step(q, kn, vn)
        np.testing.assert_allclose(out[0, 0], np.array(st["out"]), rtol=0, atol=1e-15)
        np.testing.assert_allclose(oc.seqs[0].s, np.array(st["s"]), rtol=0, atol=1e-15)
        R, ds = deltas[0]
        assert R.tolist() == list(range(oc.seqs[0].N))
