"""The seeded input generator (CPU): Philox4x32-10 known answers and shape checks."""
import numpy as np
import torch

from synth import BATCH32, TINY, normal_table, philox4x32, uniform_u16


def _ph(c, k):
    t = [torch.tensor([x], dtype=torch.int64) for x in c]
    return [int(x) for x in philox4x32(*t, k[0], k[1])]


def test_philox4x32_10_published_known_answers():
    # Known-answer vectors published with the Random123 library (Salmon et al.).
    assert _ph([0, 0, 0, 0], [0, 0]) == [0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8]
    assert _ph([0xffffffff] * 4, [0xffffffff] * 2) == [0x408f276d, 0x41c83b0e, 0xa20bc7c6, 0x6d5451fd]
    assert _ph([0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344], [0xa4093822, 0x299f31d0]) == \
        [0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1]


def test_normal_table_is_symmetric_and_increasing():
    t = normal_table().numpy().astype(np.float64)
    assert np.all(np.diff(t) > 0)
    np.testing.assert_allclose(t, -t[::-1], atol=1e-6)
    assert abs(t.mean()) < 1e-6 and abs(t.std() - 1) < 2e-3


def test_slices_equal_the_whole():
    whole = uniform_u16(9, 1, 3, torch.arange(2), 0, 1000)
    part = uniform_u16(9, 1, 3, torch.arange(2), 37, 500)
    assert torch.equal(whole[:, 37:537], part)
    k = BATCH32.kv("k", 2, 3, 0, 300)
    assert torch.equal(k[:, 100:150], BATCH32.kv("k", 2, 3, 100, 150))


def test_workload_shapes():
    assert TINY.kv_layers("k", 0, 0, 10).shape == (1, 10, 2, 64)
    lens = BATCH32.context_lens()
    assert len(lens) == 32 and min(lens) >= 1024 and max(lens) <= 8192
    assert BATCH32.queries(1).shape == (32, 28, 28, 128)
    assert TINY.spike_positions(0).numel() == 16


def test_delayed_spikes_stay_silent_until_their_group_activates():
    # The MHA configuration's delayed spikes: a spike key carries 6 sqrt(d) along its
    # group's direction e_j; a query has no component along any e_j until the
    # group's first spike is 500 positions behind it, and exactly 1 after.
    from synth import MHA16K
    w = MHA16K.replace(n_layers=1, n_q_heads=2, n_kv_heads=2, batch=1, context=("fixed", 1200),
                       prompt_len=64, key_scale=("delayed_spikes", 0.02, 6.0, 300, 4), n_steps=8)
    grp, first = w.spike_groups(0)
    assert grp.numel() > 0 and first.numel() == 4
    e = __import__("synth.workloads", fromlist=["_spike_dirs"])._spike_dirs(w, 0, 0)  # [groups, d]
    np.testing.assert_allclose((e @ e.T).numpy(), np.eye(4), atol=1e-10)
    q = w.queries(1)[0, 0, 0].to(torch.float64)            # position 1200: step 1
    pos = w.step_positions(1)[0]
    comp = (e @ q).numpy()
    active = (first + 300 <= pos).numpy()
    # the stored query is bf16: its rounding (2^-9 relative per element) bounds the error
    np.testing.assert_allclose(comp[active], 1.0, atol=2e-2)
    np.testing.assert_allclose(comp[~active], 0.0, atol=2e-2)
    # spike keys point along their group's direction, 6 sqrt(d) long beyond the noise
    spikes = w.spike_positions(0)
    k = w.kv("k", 0, 0, 0, w.total_len(0))[0].to(torch.float64)   # head 0, [n, d]
    j = int(grp[0])
    along = float(k[int(spikes[0])] @ e[j])
    assert abs(along - 6.0 * np.sqrt(w.head_dim)) < 5.0   # noise adds N(0, 1) along e_j
