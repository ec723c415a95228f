"""The debug build's device index checks, and their absence from the release
build.

The release library refuses the page-planting test hook (nothing is written)
and reports itself as no debug build. The debug library is built here and its
checks run in a child process (tests/debug_checks.py with TKV_LIB=debug), so
that this process keeps the release library.
"""
import os
import subprocess
import sys

import pytest
import torch

from helpers import prefill_cache
from synth import TINY

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_the_release_build_refuses_the_planting_hook():
    from tiered_kv_cache_split_gb300 import TieredKVCache, _lib as L
    assert not L.DEBUG and L.load().tkv_debug_build() == 0
    torch.cuda.set_device(DEV)
    c = TieredKVCache.from_workload(TINY)
    try:
        prefill_cache(c, TINY, DEV)
        with pytest.raises(L.TkvError) as err:
            c.test_plant_bad_page(0, 0, 0)
        assert err.value.status == L.ERR_STATE
        out = c.decode_step(TINY.queries(1).to(DEV), TINY.kv_new("k", 1).to(DEV), TINY.kv_new("v", 1).to(DEV))
        c.synchronize()                                  # the handle is not broken
        assert bool(torch.isfinite(out.float()).all())
    finally:
        c.close()


def test_the_debug_build_in_a_child_process():
    from tiered_kv_cache_split_gb300 import build
    lib = build.build(debug=True)
    assert lib.endswith("libtkv_debug.so")
    env = dict(os.environ, TKV_LIB="debug")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        os.path.join(HERE, "debug_checks.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert "5 passed" in r.stdout, r.stdout[-2000:]
