"""The allocation-free paged attention entry point, through the C ABI.

Some callers cannot call cudaMalloc — an inference-engine plugin whose
per-step hook must not allocate, or a process whose framework has already
reserved all device memory — so tkv_paged_attention_noalloc keeps its scratch
in a fixed array inside the library instead of a caller buffer. This test
checks, on two calls in a row (the array keeps the previous call's contents),
that it gives what tkv_paged_attention gives with a caller-provided scratch,
within the tolerances the other attention tests use, and that a shape too large
for the array is refused without a launch. It lives in its own file so that it
runs last and also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from helpers import SCORE_ATOL, SCORE_RTOL

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _inputs(rng, B, Hq, Hkv, d, counts):
    n_pages = sum(counts) + 2
    pool = torch.from_numpy(rng.standard_normal((n_pages, Hkv, 2, 16, d)).astype(np.float32))
    pool = pool.to(torch.bfloat16).to(DEV)
    perm = rng.permutation(n_pages)
    table = np.zeros((B, max(counts)), dtype=np.int32)
    at = 0
    for b, n in enumerate(counts):
        table[b, :n] = perm[at:at + n]
        at += n
    masks = np.full(n_pages, 0xFFFF, dtype=np.uint32)
    masks[perm[0]] = 0x0F0F
    q = torch.from_numpy(rng.standard_normal((B, Hq, d)).astype(np.float32)).to(torch.bfloat16).to(DEV)
    return q, pool, torch.from_numpy(table).to(DEV), torch.from_numpy(masks.view(np.int32)).to(DEV)


def _call_noalloc(lib, q, pool, table, mask, counts, out, alpha):
    B, Hq, d = q.shape
    c = np.ascontiguousarray(counts, dtype=np.int32)
    return lib.tkv_paged_attention_noalloc(B, Hq, pool.shape[1], d, 1, q.data_ptr(), pool.data_ptr(),
                                           table.data_ptr(), mask.data_ptr(), c.ctypes.data,
                                           table.shape[1], out.data_ptr(), alpha.data_ptr(),
                                           torch.cuda.current_stream(DEV).cuda_stream)


def test_noalloc_matches_caller_scratch_on_two_calls_in_a_row():
    from tiered_kv_cache_split_gb300 import _lib as L
    from tiered_kv_cache_split_gb300 import paged_attention
    lib = L.load()
    torch.cuda.set_device(DEV)
    rng = np.random.default_rng(123)
    B, Hq, Hkv, d = 3, 28, 4, 128
    for call, counts in enumerate(([40, 7, 90], [13, 64, 2])):   # two calls, different shapes
        q, pool, table, mask = _inputs(rng, B, Hq, Hkv, d, counts)
        a_ref = torch.zeros((B, Hkv, table.shape[1] * 16), dtype=torch.float32, device=DEV)
        ref = paged_attention(q, pool, table, mask, counts, alpha_sum=a_ref)
        out = torch.empty_like(q)
        a = torch.zeros_like(a_ref)
        L.check(_call_noalloc(lib, q, pool, table, mask, counts, out, a))
        torch.cuda.synchronize()
        assert torch.max(torch.abs(out.float() - ref.float())).item() <= 2e-2, f"call {call}"
        want, got = a_ref.cpu().numpy(), a.cpu().numpy()
        assert np.all(np.abs(got - want) <= SCORE_RTOL * np.abs(want) + SCORE_ATOL), f"call {call}"
        status = ctypes.c_int32(-1)
        L.check(lib.tkv_paged_attention_noalloc_status(ctypes.byref(status),
                                                       torch.cuda.current_stream(DEV).cuda_stream))
        assert status.value == 0, f"call {call}: device status {status.value}"


def test_noalloc_refuses_shapes_beyond_its_scratch():
    from tiered_kv_cache_split_gb300 import _lib as L
    lib = L.load()
    torch.cuda.set_device(DEV)
    need = ctypes.c_size_t()
    L.check(lib.tkv_paged_attention_scratch_size(64, 64, 8, 128, 60000, ctypes.byref(need)))
    assert need.value > 16 << 20
    dummy = torch.zeros(16, dtype=torch.int32, device=DEV)
    counts = np.ones(64, dtype=np.int32)
    st = lib.tkv_paged_attention_noalloc(64, 64, 8, 128, 1, dummy.data_ptr(), dummy.data_ptr(),
                                         dummy.data_ptr(), dummy.data_ptr(), counts.ctypes.data, 60000,
                                         dummy.data_ptr(), None, torch.cuda.current_stream(DEV).cuda_stream)
    assert st == L.ERR_CAPACITY
    assert b"16777216" in lib.tkv_last_error(None)
