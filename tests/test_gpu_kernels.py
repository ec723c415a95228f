"""Kernel-level parity through the stateless C-ABI entry points, plus the
generator's CPU/CUDA agreement and the bitwise form of Proposition 1.

"Not All Thoughts Need HBM": Methodology 1 (tiers, 8-bit T2), 2 (scores),
3 (Proposition 1).
"""
import numpy as np
import pytest
import torch

from helpers import OUT_ATOL, SCORE_ATOL, SCORE_RTOL
from oracle import classify as oracle_classify
from oracle import decode_attention, protected_mask, quantize_rows
from synth import BATCH32, TINY, normal_f32, uniform_u32

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def test_generator_is_bit_identical_on_cpu_and_cuda():
    a = normal_f32(5, 1, 7, torch.arange(4), 96, 40000, "cpu")
    b = normal_f32(5, 1, 7, torch.arange(4), 96, 40000, DEV).cpu()
    assert torch.equal(a, b)
    k_cpu = BATCH32.kv("k", 3, 11, 100, 900)
    k_gpu = BATCH32.kv("k", 3, 11, 100, 900, DEV).cpu()
    assert torch.equal(k_cpu.view(torch.int16), k_gpu.view(torch.int16))


@pytest.mark.parametrize("seed", range(6))
def test_classifier_is_bit_exact(seed):
    from tiered_kv_cache_split_gb300 import classify
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 6))
    stride = 3000
    s = np.zeros((B, stride))
    old = np.zeros((B, stride), dtype=np.uint8)
    params = np.zeros((B, 5), dtype=np.int64)
    want = np.zeros((B, stride), dtype=np.uint8)
    n_sink, W = int(rng.integers(0, 8)), int(rng.integers(0, 200))
    for b in range(B):
        N = int(rng.integers(1, stride + 1))
        plen = int(rng.integers(0, 300))
        if seed % 2 == 0:
            s[b, :N] = np.floor(rng.random(N) * 20) / 20          # heavy ties
        else:
            s[b, :N] = rng.random(N) * np.where(rng.random(N) < 0.1, -1.0, 1.0)
        s[b, :N][rng.random(N) < 0.05] = -0.0
        P = protected_mask(N, plen, n_sink, W)
        old[b, :N] = np.where(~P & (rng.random(N) < 0.1), 3, rng.integers(0, 3, N))
        n0, n1, n2 = (int(x) for x in rng.integers(0, N // 2 + 2, 3))
        params[b] = (N, plen, n0, n1, n2)
        want[b, :N] = oracle_classify(s[b, :N], old[b, :N], plen, n_sink, W, n0, n1, n2)
    got = classify(torch.from_numpy(s).to(DEV), torch.from_numpy(old).to(DEV), params, n_sink, W)
    got = got.cpu().numpy()
    for b in range(B):
        N = params[b, 0]
        assert np.array_equal(got[b, :N], want[b, :N]), f"request {b}"


@pytest.mark.parametrize("seed", range(4))
def test_classifier_is_bit_exact_across_many_slices(seed):
    """Long sequences span many 4096-position slices of the select; with only a
    few distinct scores the ties at each boundary cross slice borders."""
    from tiered_kv_cache_split_gb300 import classify
    rng = np.random.default_rng(100 + seed)
    B, stride = 3, 40000
    s = np.zeros((B, stride))
    old = np.zeros((B, stride), dtype=np.uint8)
    params = np.zeros((B, 5), dtype=np.int64)
    want = np.zeros((B, stride), dtype=np.uint8)
    n_sink, W = 4, int(rng.integers(0, 3000))
    for b in range(B):
        N = int(rng.integers(stride // 2, stride + 1))
        plen = int(rng.integers(0, 5000))
        s[b, :N] = rng.integers(0, 6 + 10 * seed, N) / 8.0
        P = protected_mask(N, plen, n_sink, W)
        old[b, :N] = np.where(~P & (rng.random(N) < 0.05), 3, rng.integers(0, 3, N))
        n1, n2 = int(rng.integers(0, N // 3)), int(rng.integers(0, N // 3))
        n0 = int(rng.integers(0, N // 2))
        params[b] = (N, plen, n0, n1, n2)
        want[b, :N] = oracle_classify(s[b, :N], old[b, :N], plen, n_sink, W, n0, n1, n2)
    got = classify(torch.from_numpy(s).to(DEV), torch.from_numpy(old).to(DEV), params, n_sink, W)
    got = got.cpu().numpy()
    for b in range(B):
        N = params[b, 0]
        assert np.array_equal(got[b, :N], want[b, :N]), f"request {b}"


@pytest.mark.parametrize("dtype,scale", [("bf16", "f32"), ("f32", "f32"), ("bf16", "f16"), ("f32", "f16")])
def test_quantiser_is_bit_exact(dtype, scale):
    from tiered_kv_cache_split_gb300 import quantize_rows as q_gpu
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((300, 512)) * rng.lognormal(0, 1.5, (300, 1))).astype(np.float32)
    x[5] = 0.0
    x[6, :] = np.float32(2.5)                           # x / scale ties exactly at .5 steps
    x[6, 0] = np.float32(127.0)
    tx = torch.from_numpy(x)
    if dtype == "bf16":
        tx = tx.to(torch.bfloat16)
        x = tx.float().numpy()
    codes, scales = q_gpu(tx.to(DEV), scale)
    want_c, want_s = quantize_rows(x, scale)
    assert np.array_equal(codes.cpu().numpy(), want_c)
    assert np.array_equal(scales.cpu().numpy(), want_s)


def _random_pool(rng, B, Hkv, d, pages_per_seq, dtype, nan_holes=True):
    n_pages = int(sum(pages_per_seq)) + 3
    pool = rng.standard_normal((n_pages, Hkv, 2, 16, d)).astype(np.float32)
    pool[:, :, 0] *= rng.lognormal(0, 0.7, (n_pages, 1, 16, 1)).astype(np.float32)
    perm = rng.permutation(n_pages)
    max_pages = max(pages_per_seq)
    table = np.zeros((B, max_pages), dtype=np.int32)
    masks = np.full(n_pages, 0xFFFF, dtype=np.uint32)
    at = 0
    for b, n in enumerate(pages_per_seq):
        table[b, :n] = perm[at:at + n]
        at += n
    for p in rng.choice(n_pages, size=n_pages // 3, replace=False):
        masks[p] = int(rng.integers(1, 0xFFFF))
    masks[table[0, 0]] = 0                                 # a fully empty page
    if nan_holes:
        for p in range(n_pages):
            for j in range(16):
                if not (masks[p] >> j) & 1:
                    pool[p, :, :, j, :] = np.nan
    tp = torch.from_numpy(pool)
    if dtype == "bf16":
        tp = tp.to(torch.bfloat16)
    return tp, table, masks


@pytest.mark.parametrize("dtype,G,d", [("bf16", 7, 128), ("bf16", 1, 128), ("bf16", 4, 128),
                                       ("f32", 4, 64), ("bf16", 8, 64), ("f32", 2, 128)])
def test_paged_attention_and_fused_alpha(dtype, G, d):
    from tiered_kv_cache_split_gb300 import paged_attention
    rng = np.random.default_rng(G * 100 + d)
    B, Hkv = 3, 2 if G >= 4 else 4
    Hq = Hkv * G
    counts = [37, 1, 150]
    pool, table, masks = _random_pool(rng, B, Hkv, d, counts, dtype)
    q = rng.standard_normal((B, Hq, d)).astype(np.float32)
    tq = torch.from_numpy(q).to(torch.bfloat16 if dtype == "bf16" else torch.float32)
    q = tq.float().numpy()
    pool32 = pool.float().numpy()
    alpha = torch.zeros((B, Hkv, max(counts) * 16), dtype=torch.float32, device=DEV)
    out = paged_attention(tq.to(DEV), pool.to(DEV), torch.from_numpy(table).to(DEV),
                          torch.from_numpy(masks.view(np.int32)).to(DEV), counts, alpha_sum=alpha)
    out = out.float().cpu().numpy()
    alpha = alpha.cpu().numpy()
    for b in range(B):
        pages = table[b, :counts[b]]
        K, V, slots = [], [], []
        for k, p in enumerate(pages):
            for j in range(16):
                if (masks[p] >> j) & 1:
                    K.append(pool32[p, :, 0, j])
                    V.append(pool32[p, :, 1, j])
                    slots.append(16 * k + j)
        ref, a = decode_attention(q[b], np.array(K), np.array(V))
        tol = OUT_ATOL if dtype == "bf16" else 1e-4
        assert np.max(np.abs(out[b] - ref)) <= tol
        for h in range(Hkv):
            want = a[h * G:(h + 1) * G].sum(0)
            got = alpha[b, h, slots]
            assert np.all(np.abs(got - want) <= SCORE_RTOL * want + SCORE_ATOL), (b, h)
            rest = np.setdiff1d(np.arange(counts[b] * 16), slots)
            assert np.all(alpha[b, h, rest] == 0)


@pytest.mark.parametrize("dtype,G", [("bf16", 8), ("f32", 4)])
def test_paged_attention_with_more_than_64_chunks_per_sequence(dtype, G):
    """One long sequence on one KV head is split into up to 128 chunks: the
    epilogue's global (M, Z) then reduces partials beyond its first 64 per lane
    pair, and the output merge runs over every chunk."""
    from tiered_kv_cache_split_gb300 import paged_attention
    rng = np.random.default_rng(77 + G)
    B, Hkv, d = 1, 1, 128
    Hq = Hkv * G
    counts = [1200]
    pool, table, masks = _random_pool(rng, B, Hkv, d, counts, dtype)
    q = rng.standard_normal((B, Hq, d)).astype(np.float32)
    tq = torch.from_numpy(q).to(torch.bfloat16 if dtype == "bf16" else torch.float32)
    q = tq.float().numpy()
    pool32 = pool.float().numpy()
    alpha = torch.zeros((B, Hkv, counts[0] * 16), dtype=torch.float32, device=DEV)
    out = paged_attention(tq.to(DEV), pool.to(DEV), torch.from_numpy(table).to(DEV),
                          torch.from_numpy(masks.view(np.int32)).to(DEV), counts, alpha_sum=alpha)
    out = out.float().cpu().numpy()
    alpha = alpha.cpu().numpy()
    K, V, slots = [], [], []
    for k, p in enumerate(table[0, :counts[0]]):
        for j in range(16):
            if (masks[p] >> j) & 1:
                K.append(pool32[p, :, 0, j])
                V.append(pool32[p, :, 1, j])
                slots.append(16 * k + j)
    ref, a = decode_attention(q[0], np.array(K), np.array(V))
    assert np.max(np.abs(out[0] - ref)) <= (OUT_ATOL if dtype == "bf16" else 1e-4)
    want = a.sum(0)
    got = alpha[0, 0, slots]
    assert np.all(np.abs(got - want) <= SCORE_RTOL * want + SCORE_ATOL)


def test_proposition_1_bitwise_on_the_gpu():
    """Attention over T0 + prefetched T1 gives the same bits as the same pages,
    in the same order, all resident in HBM (same kernel, same fixed chunking)."""
    from tiered_kv_cache_split_gb300 import TieredKVCache, paged_attention
    from helpers import prefill_cache
    torch.cuda.set_device(DEV)
    w = TINY
    cache = TieredKVCache.from_workload(w, budget_mode="count", budgets=(200, 1000, 0, 0))
    prefill_cache(cache, w, DEV)
    cache.set_scores(0, w.synthetic_scores(0, w.context_lens()[0]).numpy())
    cache.reclassify()
    assert (cache.tiers(0) == 1).sum() > 100 and (cache.tiers(0) >= 2).sum() == 0
    q = w.queries(1)
    out = cache.decode_step(q.to(DEV), w.kv_new("k", 1).to(DEV), w.kv_new("v", 1).to(DEV))
    torch.cuda.synchronize()
    # rebuild the exact page contents, T0 pages then T1 pages, in one HBM pool
    rows, masks = [], []
    for tier in (0, 1):
        pages, pm, pos = cache.page_table(0, tier)
        for i in range(len(pages)):
            page = np.zeros((w.n_kv_heads, 2, 16, w.head_dim), dtype=np.float32)
            for j in range(16):
                if pos[i, j] >= 0:
                    k, v = cache.kv_row(0, int(pos[i, j]))
                    page[:, 0, j] = k[0].numpy()
                    page[:, 1, j] = v[0].numpy()
            rows.append(page)
            masks.append(int(pm[i]))
    pool = torch.from_numpy(np.stack(rows)).to(DEV)
    table = torch.arange(len(rows), dtype=torch.int32, device=DEV).view(1, -1)
    mask_t = torch.tensor(masks, dtype=torch.int32, device=DEV)
    ref = paged_attention(q[0, 0].unsqueeze(0).to(DEV), pool, table, mask_t, [len(rows)])
    assert torch.equal(ref[0].cpu(), out[0, 0].cpu())
    cache.close()

