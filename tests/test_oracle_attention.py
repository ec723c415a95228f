"""Pins of the oracle's decode attention (CPU only).

"Not All Thoughts Need HBM", Methodology 3: attention over the retained tokens
is ordinary softmax attention; with nothing evicted it is exactly the
textbook single-query attention that torch's float64 SDPA computes.
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import decode_attention


def test_hand_worked_three_tokens(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "attention_3tok.json")))
    out, alpha = decode_attention(np.array(g["q"]), np.array(g["k"]), np.array(g["v"]))
    np.testing.assert_allclose(alpha, np.array(g["alpha"]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(out, np.array(g["out"]), rtol=0, atol=1e-14)


@pytest.mark.parametrize("Hq,Hkv,d,n", [(8, 2, 64, 37), (28, 4, 128, 300), (4, 4, 16, 1)])
def test_matches_torch_sdpa_when_nothing_is_evicted(Hq, Hkv, d, n):
    rng = np.random.default_rng(Hq * 1000 + n)
    q = rng.standard_normal((Hq, d))
    K = rng.standard_normal((n, Hkv, d)) * 2.0
    V = rng.standard_normal((n, Hkv, d))
    out, alpha = decode_attention(q, K, V)
    G = Hq // Hkv
    tq = torch.from_numpy(q).view(1, Hq, 1, d)
    tk = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0)
    tv = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv)
    np.testing.assert_allclose(out, ref[0, :, 0].numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(alpha.sum(1), np.ones(Hq), rtol=0, atol=1e-12)


def test_gqa_head_mapping_uses_consecutive_query_heads():
    # KV head 0 holds value +1 everywhere, KV head 1 holds -1: query heads 0, 1
    # must read +1 and heads 2, 3 must read -1 (head h -> kv head h // G).
    n, d = 5, 8
    K = np.zeros((n, 2, d))
    V = np.stack([np.ones((n, d)), -np.ones((n, d))], axis=1)
    out, _ = decode_attention(np.zeros((4, d)), K, V)
    np.testing.assert_array_equal(out[:2], np.ones((2, d)))
    np.testing.assert_array_equal(out[2:], -np.ones((2, d)))


def test_single_token_returns_its_value():
    v = np.arange(6, dtype=np.float64).reshape(1, 1, 6)
    out, alpha = decode_attention(np.ones((3, 6)), np.ones((1, 1, 6)) * 5, v)
    assert np.all(alpha == 1.0)
    np.testing.assert_array_equal(out, np.repeat(v[0], 3, axis=0))


def test_empty_retained_set_is_rejected():
    with pytest.raises(ValueError):
        decode_attention(np.ones((2, 4)), np.zeros((0, 1, 4)), np.zeros((0, 1, 4)))
