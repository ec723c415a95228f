"""Host-side fault injection: a failed call is reported, and what it promises
about the state holds.

The library's own host calls are the injection sites (tkv_test_inject_fault or
the TKV_FAULT environment variable): the workspace set-up of tkv_create, the
copies of caller data to and from the device, the T1/T2 prefetch enqueue and
the reassignment's allocator. Nothing faults, traps or hangs on the GPU.

The promises checked here:
  * a failed copy of caller inputs, score upload or read, or a reassignment
    that does not fit, changes nothing: a twin cache that never saw the failure
    keeps producing bitwise the same outputs, scores, tiers and page tables;
  * a failed output copy leaves the step in effect and the handle usable;
  * a prefetch that fails in the middle of a step breaks the handle, the work
    already enqueued drains, and the device and a fresh handle keep working;
  * a failed tkv_create leaves nothing behind, at every one of its set-up calls.
"""
import gc

import numpy as np
import pytest
import torch

from helpers import prefill_cache
from synth import CHAIN7B

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
W = CHAIN7B.replace(n_layers=4, batch=3, context=("uniform", 200, 600), prompt_len=32, recent_window=32,
                    reclassify_interval=4, n_steps=16)


def _cache(**kw):
    from tiered_kv_cache_split_gb300 import TieredKVCache
    torch.cuda.set_device(DEV)
    c = TieredKVCache.from_workload(W, layers_per_launch=2, **kw)
    prefill_cache(c, W, DEV)
    return c


def _host_inputs(t):
    return tuple(x.pin_memory() for x in (W.queries(t), W.kv_new("k", t), W.kv_new("v", t)))


def _state(c):
    st = []
    for b in range(W.batch):
        st.append((c.seq_len(b), c.scores(b).copy(), c.tiers(b).copy(),
                   [tuple(a.copy() for a in c.page_table(b, t)) for t in range(3)]))
    return st


def _assert_same_state(x, y, what):
    for b, (sx, sy) in enumerate(zip(x, y)):
        assert sx[0] == sy[0], (what, b, "length")
        assert np.array_equal(sx[1], sy[1]), (what, b, "scores")
        assert np.array_equal(sx[2], sy[2]), (what, b, "tiers")
        for t in range(3):
            for u, v in zip(sx[3][t], sy[3][t]):
                assert np.array_equal(u, v), (what, b, "page table", t)


def _expect(status, fn, *args, **kw):
    from tiered_kv_cache_split_gb300 import _lib as L
    with pytest.raises(L.TkvError) as err:
        fn(*args, **kw)
    assert err.value.status == status, str(err.value)
    return str(err.value)


def test_failed_copies_and_overflow_change_nothing():
    from tiered_kv_cache_split_gb300 import _lib as L
    a, b = _cache(), _cache()
    try:
        for t in range(1, 14):
            q, k, v = _host_inputs(t)
            if t == 2:   # second input copy of the step (the new keys)
                before = _state(b)
                b.test_inject_fault("h2d", 2)
                assert "injected" in _expect(L.ERR_CUDA, b.decode_step_host, q, k, v)
                _assert_same_state(before, _state(b), "after a failed input copy")
            if t == 3:   # a score upload that fails
                before = _state(b)
                b.test_inject_fault("h2d")
                _expect(L.ERR_CUDA, b.set_scores, 1, np.full(b.seq_len(1), 7.0))
                _assert_same_state(before, _state(b), "after a failed score upload")
            if t == 6:   # reads that fail, then succeed
                b.test_inject_fault("d2h")
                _expect(L.ERR_CUDA, b.scores, 0)
                t0 = int(np.nonzero(b.tiers(2) == 0)[0][0])
                b.test_inject_fault("d2h")
                _expect(L.ERR_CUDA, b.kv_row, 2, t0)
                ka, va = a.kv_row(2, t0)
                kb, vb = b.kv_row(2, t0)
                assert torch.equal(ka, kb) and torch.equal(va, vb)
            if t == 7:   # a reassignment that does not fit, between steps
                before = _state(b)
                b.test_inject_fault("classify_overflow")
                assert "injected" in _expect(L.ERR_CAPACITY, b.reclassify)
                _assert_same_state(before, _state(b), "after a reassignment that did not fit")
            if t == 10:  # the output copy fails: the step itself took effect on both
                b.test_inject_fault("d2h")
                _expect(L.ERR_CUDA, b.decode_step_host, q, k, v)
                a.decode_step_host(q, k, v)
                continue
            oa = a.decode_step_host(q, k, v)
            ob = b.decode_step_host(q, k, v)
            assert torch.equal(oa, ob), f"step {t}"
        _assert_same_state(_state(a), _state(b), "at the end")
        assert sum(int(np.count_nonzero(a.tiers(i) == 1)) for i in range(W.batch)) > 0  # T1 was in play
    finally:
        a.close()
        b.close()


def test_the_environment_arms_a_handle_site(monkeypatch):
    from tiered_kv_cache_split_gb300 import _lib as L
    monkeypatch.setenv("TKV_FAULT", "h2d:3")   # the third input copy: the new values
    c = _cache()
    monkeypatch.delenv("TKV_FAULT")
    try:
        q, k, v = _host_inputs(1)
        n = c.seq_len(0)
        _expect(L.ERR_CUDA, c.decode_step_host, q, k, v)
        assert c.seq_len(0) == n
        out = c.decode_step_host(q, k, v)
        assert c.seq_len(0) == n + 1 and bool(torch.isfinite(out.float()).all())
    finally:
        c.close()


def test_a_prefetch_that_fails_mid_step_breaks_only_the_handle():
    from tiered_kv_cache_split_gb300 import _lib as L
    c = _cache()
    try:
        q, k, v = (x.to(DEV) for x in _host_inputs(1))
        c.decode_step(q, k, v)
        c.synchronize()
        c.test_inject_fault("prefetch", 2)      # the second layer group's prefetch
        assert "injected" in _expect(L.ERR_CUDA, c.decode_step, q, k, v)
        _expect(L.ERR_STATE, c.synchronize)
        _expect(L.ERR_STATE, c.decode_step, q, k, v)
    finally:
        c.close()                               # drains what the half step enqueued
    torch.cuda.synchronize()
    fresh = _cache()
    try:
        out = fresh.decode_step(q, k, v)
        fresh.synchronize()
        assert bool(torch.isfinite(out.float()).all())
    finally:
        fresh.close()


@pytest.mark.parametrize("host_tiers,calls", [("stream", 15), ("mirror", 18)])
def test_a_failed_create_leaves_nothing_behind(host_tiers, calls, monkeypatch):
    from tiered_kv_cache_split_gb300 import TieredKVCache, _lib as L
    from tiered_kv_cache_split_gb300.cache import inject_create_fault
    torch.cuda.set_device(DEV)
    torch.cuda.synchronize()
    gc.collect()
    base = torch.cuda.memory_allocated(DEV)
    for n in range(1, calls + 1):            # every set-up call in turn
        inject_create_fault(n)
        msg = _expect(L.ERR_CUDA, TieredKVCache.from_workload, W, host_tiers=host_tiers)
        assert "injected" in msg, (n, msg)
        gc.collect()
        assert torch.cuda.memory_allocated(DEV) == base, n
    inject_create_fault(calls + 1)              # one beyond the last set-up call: never fires, dropped
    c = TieredKVCache.from_workload(W, host_tiers=host_tiers)
    c.close()
    monkeypatch.setenv("TKV_FAULT", "alloc:4")
    _expect(L.ERR_CUDA, TieredKVCache.from_workload, W, host_tiers=host_tiers)
    monkeypatch.delenv("TKV_FAULT")
    c = TieredKVCache.from_workload(W, host_tiers=host_tiers)   # nothing stays armed
    prefill_cache(c, W, DEV)
    q, k, v = (x.to(DEV) for x in _host_inputs(1))
    out = c.decode_step(q, k, v)
    c.synchronize()
    assert bool(torch.isfinite(out.float()).all())
    c.close()
