"""Checks of the debug build (libtkv_debug.so, compiled with TKV_DEBUG).

Not collected by the main suite (no test_ prefix): test_gpu_debug_build.py
builds the debug library and runs this file in a child process with
TKV_LIB=debug, so that the process loads that library instead of libtkv.so.

  * the debug build gives the same results as the oracle (its index checks
    change no arithmetic) in every host-tier mode;
  * a page id outside its pool, planted in the device page table of T0, T1 or
    T2, is caught by the attention kernel's check at the next step: the access
    is skipped, TKV_ERR_INTERNAL names the check, the id and its bound, the
    handle is broken, and a fresh handle works. The planted id is the pool's
    capacity, one past its end, whose addresses lie inside the workspace, so
    even a missed check would read allocated memory.
"""
import numpy as np
import pytest
import torch

from helpers import prefill_cache
from synth import CHAIN7B, TINY
from test_gpu_modes import _lockstep

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
W = CHAIN7B.replace(n_layers=3, batch=4, context=("uniform", 100, 500), prompt_len=16, recent_window=24,
                    reclassify_interval=4, n_steps=12)


def test_the_debug_library_is_loaded():
    from tiered_kv_cache_split_gb300 import _lib as L
    assert L.DEBUG and L.LIB_PATH.endswith("libtkv_debug.so")
    assert L.load().tkv_debug_build() == 1


def test_the_debug_build_matches_the_oracle():
    oc, _ = _lockstep(W, 10, [("stream", 0), ("mirror", 1), ("zerocopy", 3)])
    counts = np.bincount(np.concatenate([oc.seqs[b].tier for b in range(W.batch)]), minlength=4)
    assert np.all(counts > 0), counts
    _lockstep(TINY.replace(n_steps=6), 6, [("stream", 0)])


@pytest.mark.parametrize("tier", [0, 1, 2])
def test_a_page_id_outside_its_pool_is_caught(tier):
    from tiered_kv_cache_split_gb300 import TieredKVCache, _lib as L
    torch.cuda.set_device(DEV)
    args = lambda t: (W.queries(t).to(DEV), W.kv_new("k", t).to(DEV), W.kv_new("v", t).to(DEV))
    c = TieredKVCache.from_workload(W)
    try:
        prefill_cache(c, W, DEV)
        for t in range(1, W.reclassify_interval + 1):   # through the first reassignment
            c.decode_step(*args(t))
        c.synchronize()
        b = next(b for b in range(W.batch) if len(c.page_table(b, tier)[0]) > 0)
        planted = c.test_plant_bad_page(b, tier, 0)
        c.decode_step(*args(W.reclassify_interval + 1))
        with pytest.raises(L.TkvError) as err:
            c.synchronize()
        assert err.value.status == L.ERR_INTERNAL
        assert f"attention page id {planted} outside [0, {planted})" in str(err.value), str(err.value)
        with pytest.raises(L.TkvError) as err:
            c.synchronize()
        assert err.value.status == L.ERR_STATE
    finally:
        c.close()
    torch.cuda.synchronize()
    fresh = TieredKVCache.from_workload(W)
    try:
        prefill_cache(fresh, W, DEV)
        out = fresh.decode_step(*args(1))
        fresh.synchronize()
        assert bool(torch.isfinite(out.float()).all())
    finally:
        fresh.close()
