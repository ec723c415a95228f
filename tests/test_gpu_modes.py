"""Where attention finds the host tiers, and how many layers one launch covers,
must not change a single output bit.

"Not All Thoughts Need HBM", Methodology 3 (Proposition 1: T1 read at full
precision contributes exactly what it would from HBM) and Methodology 4 (T1 is
prefetched before attention; only newly promoted tokens need to move). The
same decode steps run side by side through:
  * STREAM   a per-step copy of each layer group's T1 / T2 pages into staging,
  * MIRROR   device-resident copies of the host tiers, updated differentially,
  * ZEROCOPY attention reading T1 / T2 pages in place in pinned host memory,
with 1, several, a ragged number or all layers per attention launch. Every
output must be bitwise equal to the first configuration's, every step must
match the oracle (outputs 2e-2 absolute, scores 1e-4 relative), and tiers,
page tables, 8-bit codes and the values T0/T1 tokens hold must be identical.
"""
import numpy as np
import pytest
import torch

from helpers import OUT_ATOL, assert_page_tables_equal, assert_scores_close, prefill_cache, prefill_oracle
from oracle import OracleCache
from oracle.classify import T2
from synth import CHAIN7B, MHA16K, TINY

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _lockstep(w, steps, configs, **kw):
    from tiered_kv_cache_split_gb300 import TieredKVCache
    torch.cuda.set_device(DEV)
    caches = []
    for mode, lpl in configs:
        c = TieredKVCache.from_workload(w, host_tiers=mode, layers_per_launch=lpl, **kw)
        prefill_cache(c, w, DEV)
        caches.append(c)
    oc = OracleCache.from_workload(w)
    prefill_oracle(oc, w)
    for t in range(1, steps + 1):
        q, kn, vn = w.queries(t), w.kv_new("k", t), w.kv_new("v", t)
        outs = [c.decode_step(q.to(DEV), kn.to(DEV), vn.to(DEV)) for c in caches]
        ref, _ = oc.decode_step(q.float().numpy(), kn.float().numpy(), vn.float().numpy())
        torch.cuda.synchronize()
        err = float(np.max(np.abs(outs[0].float().cpu().numpy() - ref)))
        assert err <= OUT_ATOL, f"step {t}: output error {err}"
        for i, o in enumerate(outs[1:], start=1):
            assert torch.equal(o.cpu(), outs[0].cpu()), f"step {t}: {configs[i]} differs from {configs[0]}"
        for b in range(w.batch):
            for c in caches:
                assert np.array_equal(c.tiers(b), oc.seqs[b].tier), f"step {t}: tiers of request {b}"
                assert_scores_close(c.scores(b), oc.seqs[b].s, f"step {t} request {b}")
        if t % w.reclassify_interval == 0:
            for b in range(w.batch):
                sq = oc.seqs[b]
                for c in caches:
                    assert_page_tables_equal(c, oc, b, f"step {t}")
                for pos in np.nonzero(sq.tier == T2)[0][::5]:
                    kc, ks, vc, vs = sq.codes[int(pos)]
                    for c in caches:
                        codes, scales = c.t2_row(b, int(pos))
                        assert np.array_equal(codes[:, 0], kc) and np.array_equal(codes[:, 1], vc)
                        assert np.array_equal(scales[:, 0], ks) and np.array_equal(scales[:, 1], vs)
                for pos in np.nonzero(sq.tier <= 1)[0][::11]:
                    for c in caches:
                        k, v = c.kv_row(b, int(pos))
                        assert np.array_equal(k.numpy().astype(np.float64), sq.K[:, pos]), f"K row {pos}"
                        assert np.array_equal(v.numpy().astype(np.float64), sq.V[:, pos]), f"V row {pos}"
    stats = [c.stats() for c in caches]
    for c in caches:
        c.close()
    return oc, stats


def test_chain7b_shape_in_every_host_tier_mode_and_layer_grouping():
    # 28 layers, 28 query / 4 KV heads (the tensor-core kernel), bf16; a short
    # prompt and window and Delta = 16, so that all four tiers exist from the
    # first reassignment on and tokens move between them every 16 steps.
    w = CHAIN7B.replace(context=("fixed", 600), prompt_len=64, recent_window=32, reclassify_interval=16,
                        n_steps=48)
    configs = [("stream", 1), ("stream", 0), ("mirror", 7), ("zerocopy", 28), ("mirror", 3), ("zerocopy", 0)]
    oc, stats = _lockstep(w, 48, configs)
    counts = np.bincount(oc.seqs[0].tier, minlength=4)
    assert np.all(counts > 0), counts
    launches = [s["attn_launches"] for s in stats]
    # the automatic grouping takes 14 layers per launch here: one layer's K and V are small
    assert launches == [48 * 28, 48 * 2, 48 * 4, 48 * 1, 48 * 10, 48 * 2], launches
    # per-step copies only in STREAM mode; a mirror moves T1 / T2 sources on the device
    assert stats[0]["prefetch_bytes"] > 0 and stats[2]["prefetch_bytes"] == 0 and stats[3]["prefetch_bytes"] == 0
    assert stats[2]["h2d_move_bytes"] == 0 and stats[0]["h2d_move_bytes"] > 0
    assert stats[2]["d2h_move_bytes"] == stats[0]["d2h_move_bytes"]


def test_tiny_fp32_in_every_host_tier_mode():
    _lockstep(TINY, TINY.n_steps, [("stream", 0), ("mirror", 0), ("zerocopy", 0)])


def test_mha_shape_in_every_host_tier_mode():
    # one query head per KV head (the FMA kernel), 8-bit T2 with one float16
    # scale per token and KV head, read in place from host memory in ZEROCOPY
    w = MHA16K.replace(n_layers=4, batch=2, context=("fixed", 700), prompt_len=64,
                       key_scale=("delayed_spikes", 0.02, 6.0, 40, 4), reclassify_interval=16, n_steps=32)
    _lockstep(w, 32, [("stream", 0), ("mirror", 2), ("zerocopy", 4), ("stream", 3)])


def test_full_cache_eviction_only_and_hbm_ratio_budgets():
    # the policy variants the pages measure (full cache; eviction without
    # offload; the share of HBM at fixed eviction) through the same kernels
    base = CHAIN7B.replace(n_layers=4, context=("fixed", 500), prompt_len=32, recent_window=32,
                           reclassify_interval=8, n_steps=24)
    for budgets in ((100, 0, 0, 0), (50, 0, 0, 50), (30, 50, 10, 10), (70, 10, 10, 10)):
        w = base.replace(budgets=budgets)
        oc, _ = _lockstep(w, 24, [("stream", 0), ("mirror", 0)])
        counts = np.bincount(oc.seqs[0].tier, minlength=4)
        for k in range(1, 4):
            assert (counts[k] > 0) == (budgets[k] > 0), (budgets, counts)


def test_proposition_1_bitwise_on_the_tensor_core_path():
    """bf16, 28 query / 4 KV heads: attention over T0 + prefetched T1 gives the
    same bits as the same pages, in the same order, all resident in HBM."""
    from tiered_kv_cache_split_gb300 import TieredKVCache, paged_attention
    torch.cuda.set_device(DEV)
    w = CHAIN7B.replace(context=("fixed", 700), prompt_len=64, n_steps=4)
    cache = TieredKVCache.from_workload(w, budget_mode="count", budgets=(250, 10000, 0, 0))
    prefill_cache(cache, w, DEV)
    cache.set_scores(0, w.synthetic_scores(0, w.context_lens()[0]).numpy())
    cache.reclassify()
    tiers = cache.tiers(0)
    assert (tiers == 1).sum() > 300 and (tiers >= 2).sum() == 0
    q = w.queries(1)
    out = cache.decode_step(q.to(DEV), w.kv_new("k", 1).to(DEV), w.kv_new("v", 1).to(DEV))
    torch.cuda.synchronize()
    layout = []  # (positions of each page's slots, mask), T0 pages then T1 pages
    for tier in (0, 1):
        pages, pm, pos = cache.page_table(0, tier)
        for i in range(len(pages)):
            layout.append((pos[i], int(pm[i])))
    rows = {int(p): cache.kv_row(0, int(p)) for pos, _ in layout for p in pos if p >= 0}
    for layer in (0, 13, 27):
        pool = np.zeros((len(layout), w.n_kv_heads, 2, 16, w.head_dim), dtype=np.float32)
        for i, (pos, _) in enumerate(layout):
            for j in range(16):
                if pos[j] >= 0:
                    k, v = rows[int(pos[j])]
                    pool[i, :, 0, j] = k[layer].numpy()
                    pool[i, :, 1, j] = v[layer].numpy()
        tp = torch.from_numpy(pool).to(torch.bfloat16).to(DEV)
        table = torch.arange(len(layout), dtype=torch.int32, device=DEV).view(1, -1)
        mask_t = torch.tensor([m for _, m in layout], dtype=torch.int32, device=DEV)
        ref = paged_attention(q[0, layer].unsqueeze(0).to(DEV), tp, table, mask_t, [len(layout)])
        assert torch.equal(ref[0].cpu(), out[0, layer].cpu()), f"layer {layer}"
    cache.close()


def test_sixty_four_sequences_of_ragged_tiny_lengths():
    # the batch limit (64 sequences), a one-token sequence and lengths around page
    # boundaries, eight query heads per KV head at d = 64 (the tensor-core kernel's
    # G = 8 variant), counted budgets so that even the shortest sequences tier
    w = CHAIN7B.replace(n_layers=3, n_q_heads=16, n_kv_heads=2, head_dim=64, batch=64,
                        context=("uniform", 1, 90), prompt_len=4, n_sink=2, recent_window=3,
                        budget_mode="count", budgets=(12, 20, 8, 0), reclassify_interval=4, n_steps=12)
    lens = w.context_lens()
    assert min(lens) <= 3 and max(lens) >= 60
    oc, stats = _lockstep(w, 12, [("stream", 0), ("mirror", 2), ("zerocopy", 1)])
    counts = np.bincount(np.concatenate([oc.seqs[b].tier for b in range(w.batch)]), minlength=4)
    assert np.all(counts > 0), counts
