"""The C-ABI library loads and exports every entry point include/tkv.h
declares; host-only calls validate their arguments (CPU, no CUDA device)."""
import ctypes
import os
import re

import pytest

from tiered_kv_cache_split_gb300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "tkv.h")).read()
    return sorted(set(re.findall(r"^TKV_API [^;(]*?\b(tkv_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(L.LIB_PATH):
        from tiered_kv_cache_split_gb300 import build
        build.build()
    return L.load()


def test_every_declared_symbol_is_exported(lib):
    declared = _declared()
    assert len(declared) >= 20
    for name in declared:
        assert hasattr(lib, name), name
    assert declared == L.exported_symbols()


def _cfg(**kw):
    c = L.Config()
    c.n_layers, c.n_q_heads, c.n_kv_heads, c.head_dim = 28, 28, 4, 128
    c.kv_dtype, c.max_batch, c.max_tokens, c.page_size = L.DTYPE_BF16, 32, 8448, 16
    c.n_sink, c.recent_window, c.budget_mode = 4, 128, L.BUDGET_PERCENT
    for i, b in enumerate((40, 40, 10, 10)):
        c.budget[i] = b
    c.reclassify_interval = 64
    c.t2_scale_gran, c.t2_scale_dtype = L.SCALE_PER_TOKEN, L.SCALE_F32
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def test_workspace_size_of_the_batch32_shape(lib):
    d, p = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.tkv_workspace_size(ctypes.byref(_cfg()), ctypes.byref(d), ctypes.byref(p)) == L.OK
    kv_total = 32 * 8448 * 28 * 4 * 2 * 128 * 2      # every token can start in T0
    assert d.value > kv_total and p.value > 0.4 * kv_total


@pytest.mark.parametrize("field,value", [("page_size", 32), ("n_q_heads", 30), ("head_dim", 96),
                                         ("max_batch", 65), ("reclassify_interval", 0),
                                         ("t2_scale_dtype", L.SCALE_F16), ("budget_mode", 7)])
def test_invalid_configs_are_rejected_with_a_message(lib, field, value):
    d, p = ctypes.c_size_t(), ctypes.c_size_t()
    st = lib.tkv_workspace_size(ctypes.byref(_cfg(**{field: value})), ctypes.byref(d), ctypes.byref(p))
    assert st == L.ERR_INVALID_ARG
    assert b"invalid config" in lib.tkv_last_error(None)


def test_percent_budgets_must_sum_to_100(lib):
    c = _cfg()
    c.budget[3] = 11
    assert lib.tkv_workspace_size(ctypes.byref(c), ctypes.byref(ctypes.c_size_t()),
                                  ctypes.byref(ctypes.c_size_t())) == L.ERR_INVALID_ARG


def test_create_refuses_null_or_small_workspaces(lib):
    h = ctypes.c_void_p()
    st = lib.tkv_create(ctypes.byref(_cfg()), None, 0, None, 0, None, None, ctypes.byref(h))
    assert st == L.ERR_INVALID_ARG and not h.value
    buf = (ctypes.c_char * 4096)()
    addr = (ctypes.addressof(buf) + 255) // 256 * 256
    st = lib.tkv_create(ctypes.byref(_cfg()), addr, 1024, addr, 1024, None, None, ctypes.byref(h))
    assert st == L.ERR_CAPACITY and b"too small" in lib.tkv_last_error(None)


def test_null_handle_calls_fail_cleanly(lib):
    assert lib.tkv_reclassify(None) == L.ERR_INVALID_ARG
    assert lib.tkv_destroy(None) == L.OK
    assert lib.tkv_last_error(None)


def test_stateless_shape_checks(lib):
    n = ctypes.c_size_t()
    assert lib.tkv_paged_attention_scratch_size(2, 28, 4, 128, 100, ctypes.byref(n)) == L.OK and n.value > 0
    assert lib.tkv_paged_attention_scratch_size(2, 30, 4, 128, 100, ctypes.byref(n)) == L.ERR_INVALID_ARG
    assert lib.tkv_classify_scratch_size(4, 1000, ctypes.byref(n)) == L.OK and n.value >= 32000
    assert lib.tkv_quantize_rows(None, 1, 1, 8, None, None, 0, None) == L.ERR_INVALID_ARG


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_workspace_by_host_tier_mode(lib, mode):
    """STREAM holds a two-slot staging ring of layer groups, MIRROR a device copy
    of every layer of T1 / T2, ZEROCOPY neither; the pinned pools are the same."""
    d, p = ctypes.c_size_t(), ctypes.c_size_t()
    base_d, base_p = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.tkv_workspace_size(ctypes.byref(_cfg(host_tiers=2, layers_per_launch=4)), ctypes.byref(base_d),
                                  ctypes.byref(base_p)) == L.OK
    assert lib.tkv_workspace_size(ctypes.byref(_cfg(host_tiers=mode, layers_per_launch=4)), ctypes.byref(d),
                                  ctypes.byref(p)) == L.OK
    assert p.value == base_p.value
    t1_layer = (32 * (40 * 8448 // 100 // 16 + 2)) * 4 * 2 * 16 * 128 * 2   # about one layer of the T1 pool
    if mode == 0:
        assert 2 * 4 * 0.9 * t1_layer < d.value - base_d.value < 2 * 4 * 1.5 * t1_layer
    elif mode == 1:
        assert 28 * 0.9 * t1_layer < d.value - base_d.value < 28 * 1.5 * t1_layer
    else:
        assert d.value == base_d.value


@pytest.mark.parametrize("field,value", [("host_tiers", 3), ("layers_per_launch", -1)])
def test_invalid_mode_fields_are_rejected(lib, field, value):
    d, p = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.tkv_workspace_size(ctypes.byref(_cfg(**{field: value})), ctypes.byref(d), ctypes.byref(p)) == L.ERR_INVALID_ARG
    assert field.encode() in lib.tkv_last_error(None)


def test_test_hook_and_status_calls_fail_cleanly_without_a_handle(lib):
    assert lib.tkv_test_stall_next_attention(None, 5_000_000) == L.ERR_INVALID_ARG
    assert lib.tkv_paged_attention_noalloc_status(None, None) == L.ERR_INVALID_ARG


def test_fault_injection_arguments_are_checked_without_a_device(lib):
    F = L.FAULT_SITES
    assert lib.tkv_test_inject_fault(None, 9, 1) == L.ERR_INVALID_ARG           # unknown site
    assert lib.tkv_test_inject_fault(None, -1, 1) == L.ERR_INVALID_ARG
    assert lib.tkv_test_inject_fault(None, F["alloc"], 0) == L.ERR_INVALID_ARG  # countdown < 1
    for site in ("h2d", "d2h", "prefetch", "classify_overflow"):               # need a handle
        assert lib.tkv_test_inject_fault(None, F[site], 1) == L.ERR_INVALID_ARG
        assert b"null handle" in lib.tkv_last_error(None)
    # the allocation site is process-wide: arming and disarming touch no device
    assert lib.tkv_test_inject_fault(None, F["alloc"], 3) == L.OK
    assert lib.tkv_test_inject_fault(None, F["none"], 0) == L.OK


def test_the_release_library_has_no_index_checks(lib):
    assert lib.tkv_debug_build() == 0
    planted = ctypes.c_int32(-7)
    assert lib.tkv_test_plant_bad_page(None, 0, 1, 0, ctypes.byref(planted)) == L.ERR_INVALID_ARG
    assert planted.value == -7
