"""Pins of the oracle's cumulative-score increment (CPU only).

"Not All Thoughts Need HBM", Methodology 2: s_i grows by the attention weight
averaged over heads and then over layers.
"""
import json
import os

import numpy as np

from oracle import decode_attention, score_increment


def test_hand_worked_two_layers_two_heads(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "score_2x2.json")))
    ds = score_increment([np.array(a) for a in g["alphas"]])
    np.testing.assert_allclose(ds, g["delta"], rtol=0, atol=1e-15)


def test_increments_of_one_step_sum_to_one():
    rng = np.random.default_rng(7)
    n, L, Hq, Hkv, d = 50, 3, 6, 2, 16
    K = rng.standard_normal((L, n, Hkv, d)) * 3
    V = rng.standard_normal((L, n, Hkv, d))
    alphas = [decode_attention(rng.standard_normal((Hq, d)), K[l], V[l])[1] for l in range(L)]
    ds = score_increment(alphas)
    assert abs(ds.sum() - 1.0) < 1e-12
    assert np.all(ds >= 0)


def test_one_layer_one_head_is_that_heads_attention_row():
    # H2O-style cumulative attention: with |L| = H = 1 the increment is alpha.
    a = np.array([[0.1, 0.2, 0.7]])
    np.testing.assert_array_equal(score_increment([a]), a[0])


def test_heads_are_averaged_not_summed():
    a = np.array([[1.0, 0.0], [0.0, 1.0], [0.0, 1.0], [0.0, 1.0]])
    np.testing.assert_allclose(score_increment([a]), [0.25, 0.75], atol=1e-15)
