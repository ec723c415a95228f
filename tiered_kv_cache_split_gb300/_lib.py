"""ctypes declarations of the C ABI in include/tkv.h (argument marshalling only).

Loading fails loudly when libtkv.so has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# TKV_LIB=debug selects the debug build (device index checks; build(debug=True))
DEBUG = os.environ.get("TKV_LIB", "") == "debug"
LIB_PATH = os.path.join(HERE, "libtkv_debug.so" if DEBUG else "libtkv.so")

OK, ERR_INVALID_ARG, ERR_CAPACITY, ERR_STATE, ERR_CUDA, ERR_TIMEOUT, ERR_INTERNAL = range(7)
STATUS_NAMES = ["OK", "INVALID_ARG", "CAPACITY", "STATE", "CUDA", "TIMEOUT", "INTERNAL"]
DTYPE_F32, DTYPE_BF16 = 0, 1
BUDGET_PERCENT, BUDGET_COUNT = 0, 1
SCALE_PER_TOKEN, SCALE_PER_TOKEN_HEAD = 0, 1
SCALE_F32, SCALE_F16 = 0, 1
T2_ATTEND, T2_MASK = 0, 1
HOST_TIERS = {"stream": 0, "mirror": 1, "zerocopy": 2}
FLAG_TIMING = 1
FAULT_SITES = {"none": 0, "alloc": 1, "h2d": 2, "d2h": 3, "prefetch": 4, "classify_overflow": 5}

c_i32, c_i64, c_sz, c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p


class Config(ctypes.Structure):
    _fields_ = [
        ("n_layers", c_i32), ("n_q_heads", c_i32), ("n_kv_heads", c_i32), ("head_dim", c_i32),
        ("kv_dtype", c_i32), ("max_batch", c_i32), ("max_tokens", c_i64), ("page_size", c_i32),
        ("n_sink", c_i32), ("recent_window", c_i32), ("budget_mode", c_i32),
        ("budget", c_i64 * 4), ("reclassify_interval", c_i32), ("t2_scale_gran", c_i32),
        ("t2_scale_dtype", c_i32), ("t2_mode", c_i32), ("t0_pages", c_i64), ("t1_pages", c_i64),
        ("t2_pages", c_i64), ("max_staged_movers", c_i64), ("split_pages", c_i32), ("flags", c_i32),
        ("host_tiers", c_i32), ("layers_per_launch", c_i32),
    ]


class Stats(ctypes.Structure):
    _fields_ = [
        ("steps", c_i64), ("reclassifies", c_i64), ("movers", c_i64), ("attn_launches", c_i64),
        ("attn_bytes", c_i64), ("prefetch_bytes", c_i64), ("h2d_move_bytes", c_i64),
        ("d2h_move_bytes", c_i64), ("tier_counts", c_i64 * 4), ("attn_ms", ctypes.c_double),
        ("combine_ms", ctypes.c_double),
        ("prefetch_ms", ctypes.c_double), ("reclassify_ms", ctypes.c_double),
        ("kernel_launches", c_i64), ("attn_span_ms", ctypes.c_double), ("attn_layers", c_i64),
        ("classify_ms", ctypes.c_double), ("allocate_ms", ctypes.c_double), ("move_ms", ctypes.c_double),
    ]


class TkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"tkv {name}: {message}")


_SIGS = {
    "tkv_workspace_size": [ctypes.POINTER(Config), ctypes.POINTER(c_sz), ctypes.POINTER(c_sz)],
    "tkv_create": [ctypes.POINTER(Config), c_vp, c_sz, c_vp, c_sz, c_vp, c_vp, ctypes.POINTER(c_vp)],
    "tkv_destroy": [c_vp],
    "tkv_append": [c_vp, c_i32, c_vp, c_vp, c_i64, c_i32],
    "tkv_decode_step": [c_vp, c_vp, c_vp, c_vp, c_vp],
    "tkv_decode_step_host": [c_vp, c_vp, c_vp, c_vp, c_vp],
    "tkv_reclassify": [c_vp],
    "tkv_prefetch": [c_vp, c_i32, c_i32],
    "tkv_synchronize": [c_vp],
    "tkv_num_sequences": [c_vp, ctypes.POINTER(c_i32)],
    "tkv_seq_len": [c_vp, c_i32, ctypes.POINTER(c_i64)],
    "tkv_get_scores": [c_vp, c_i32, c_vp, c_i64],
    "tkv_set_scores": [c_vp, c_i32, c_vp, c_i64],
    "tkv_get_tiers": [c_vp, c_i32, c_vp, c_i64],
    "tkv_get_page_table": [c_vp, c_i32, c_i32, c_vp, c_vp, c_vp, c_i64, ctypes.POINTER(c_i64)],
    "tkv_get_t2_row": [c_vp, c_i32, c_i64, c_vp, c_vp],
    "tkv_get_kv_row": [c_vp, c_i32, c_i64, c_vp, c_vp],
    "tkv_get_stats": [c_vp, ctypes.POINTER(Stats)],
    "tkv_reset_stats": [c_vp],
    "tkv_paged_attention_scratch_size": [c_i32, c_i32, c_i32, c_i32, c_i32, ctypes.POINTER(c_sz)],
    "tkv_paged_attention": [c_i32, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32,
                            c_vp, c_vp, c_vp, c_sz, c_vp],
    "tkv_paged_attention_noalloc": [c_i32, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32,
                                    c_vp, c_vp, c_vp],
    "tkv_paged_attention_noalloc_status": [ctypes.POINTER(c_i32), c_vp],
    "tkv_test_stall_next_attention": [c_vp, ctypes.c_uint64],
    "tkv_test_inject_fault": [c_vp, c_i32, c_i32],
    "tkv_test_plan_attention": [c_i32, c_vp, c_vp, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp, ctypes.POINTER(c_i32)],
    "tkv_test_plant_bad_page": [c_vp, c_i32, c_i32, c_i64, ctypes.POINTER(c_i32)],
    "tkv_classify_scratch_size": [c_i32, c_i64, ctypes.POINTER(c_sz)],
    "tkv_classify": [c_i32, c_vp, c_vp, c_vp, c_i64, c_vp, c_i32, c_i32, c_vp, c_sz, c_vp],
    "tkv_quantize_rows": [c_vp, c_i32, c_i64, c_i32, c_vp, c_vp, c_i32, c_vp],
}

_lib = None


def load() -> ctypes.CDLL:
    """The loaded libtkv.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it first "
                          "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    for name, args in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.tkv_last_error.argtypes = [c_vp]
    lib.tkv_last_error.restype = ctypes.c_char_p
    lib.tkv_debug_build.argtypes = []
    lib.tkv_debug_build.restype = c_i32
    _lib = lib
    return lib


def check(status: int, handle=None) -> None:
    if status != OK:
        msg = load().tkv_last_error(handle)
        raise TkvError(status, msg.decode() if msg else "")


def exported_symbols() -> list[str]:
    return sorted(list(_SIGS) + ["tkv_last_error", "tkv_debug_build"])
