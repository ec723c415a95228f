"""A bounded device wait that runs out is reported, not hung on.

Every wait inside the attention kernels (a consumer waiting for a page, the
producer waiting for a free stage, the drain after an abort) gives up after a
time limit. Here a test hook makes one CTA withhold its first page copy, so a
consumer's wait runs out: nothing is in flight for that stage, the CTA lands
every other copy it issued and publishes an empty partial, and the host sees
TKV_ERR_TIMEOUT at the next synchronising call. The handle is then broken; the
device and a fresh handle keep working.
"""
import pytest
import torch

from helpers import prefill_cache
from synth import CHAIN7B, TINY

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.mark.parametrize("w", [TINY, CHAIN7B.replace(n_layers=2, context=("fixed", 400), n_steps=4)],
                         ids=["fp32_fma", "bf16_mma"])
def test_a_withheld_page_times_out_and_breaks_only_the_handle(w):
    from tiered_kv_cache_split_gb300 import TieredKVCache, _lib as L
    torch.cuda.set_device(DEV)
    cache = TieredKVCache.from_workload(w)
    prefill_cache(cache, w, DEV)
    args = lambda t: (w.queries(t).to(DEV), w.kv_new("k", t).to(DEV), w.kv_new("v", t).to(DEV))
    cache.decode_step(*args(1))
    cache.synchronize()
    cache.test_stall_next_attention(5_000_000)          # 5 ms limit
    cache.decode_step(*args(2))                          # enqueues; the kernel gives up by itself
    with pytest.raises(L.TkvError) as err:
        cache.synchronize()
    assert err.value.status == L.ERR_TIMEOUT
    with pytest.raises(L.TkvError) as err:
        cache.decode_step(*args(3))
    assert err.value.status == L.ERR_STATE                # broken from now on
    cache.close()
    # the device context is intact: a fresh handle runs a step
    torch.cuda.synchronize()
    fresh = TieredKVCache.from_workload(w)
    prefill_cache(fresh, w, DEV)
    out = fresh.decode_step(*args(1))
    fresh.synchronize()
    assert bool(torch.isfinite(out.float()).all())
    fresh.close()
