"""Python face of libtkv: PyTorch allocates the workspaces and streams and the
C ABI does every step of the decode path in CUDA kernels.

Methods map one to one onto include/tkv.h; nothing here computes attention,
scores, tiers or codes.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _lib as L

_DT = {"f32": L.DTYPE_F32, "bf16": L.DTYPE_BF16}
_TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def _ptr(t: torch.Tensor) -> int:
    return t.data_ptr()


class TieredKVCache:
    """A four-tier KV cache with its decode step on one CUDA device."""

    def __init__(self, *, n_layers, n_q_heads, n_kv_heads, head_dim, kv_dtype="bf16", max_batch=1,
                 max_tokens=4096, n_sink=4, recent_window=128, budget_mode="percent",
                 budgets=(50, 30, 10, 10), reclassify_interval=64, t2_scale_gran="token",
                 t2_scale_dtype="f32", t2_mode="attend", t0_pages=0, t1_pages=0, t2_pages=0,
                 max_staged_movers=0, split_pages=0, timing=False, host_tiers="stream",
                 layers_per_launch=0, device="cuda"):
        self.lib = L.load()
        self.device = torch.device(device)
        self.kv_dtype = kv_dtype
        self.torch_dtype = _TORCH_DT[kv_dtype]
        self.shape = (n_layers, n_q_heads, n_kv_heads, head_dim)
        self.t2_scale_gran = t2_scale_gran
        cfg = L.Config()
        cfg.n_layers, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim = n_layers, n_q_heads, n_kv_heads, head_dim
        cfg.kv_dtype = _DT[kv_dtype]
        cfg.max_batch = max_batch
        cfg.max_tokens = max_tokens
        cfg.page_size = 16
        cfg.n_sink, cfg.recent_window = n_sink, recent_window
        cfg.budget_mode = L.BUDGET_PERCENT if budget_mode == "percent" else L.BUDGET_COUNT
        for i, b in enumerate(budgets):
            cfg.budget[i] = int(b)
        cfg.reclassify_interval = reclassify_interval
        cfg.t2_scale_gran = L.SCALE_PER_TOKEN if t2_scale_gran == "token" else L.SCALE_PER_TOKEN_HEAD
        cfg.t2_scale_dtype = L.SCALE_F32 if t2_scale_dtype == "f32" else L.SCALE_F16
        cfg.t2_mode = L.T2_ATTEND if t2_mode == "attend" else L.T2_MASK
        cfg.t0_pages, cfg.t1_pages, cfg.t2_pages = t0_pages, t1_pages, t2_pages
        cfg.max_staged_movers = max_staged_movers
        cfg.split_pages = split_pages
        cfg.flags = L.FLAG_TIMING if timing else 0
        cfg.host_tiers = L.HOST_TIERS[host_tiers]
        cfg.layers_per_launch = layers_per_launch
        self.cfg = cfg
        dev_b, pin_b = ctypes.c_size_t(), ctypes.c_size_t()
        L.check(self.lib.tkv_workspace_size(ctypes.byref(cfg), ctypes.byref(dev_b), ctypes.byref(pin_b)))
        self.dev_bytes, self.pinned_bytes = dev_b.value, pin_b.value
        with torch.cuda.device(self.device):
            self._dev = torch.empty(self.dev_bytes, dtype=torch.uint8, device=self.device)
            self._pin = torch.empty(self.pinned_bytes, dtype=torch.uint8, pin_memory=True)
            self.compute = torch.cuda.Stream(self.device)
            self.copy = torch.cuda.Stream(self.device)
            h = ctypes.c_void_p()
            L.check(self.lib.tkv_create(ctypes.byref(cfg), _ptr(self._dev), self.dev_bytes, _ptr(self._pin),
                                        self.pinned_bytes, self.compute.cuda_stream, self.copy.cuda_stream,
                                        ctypes.byref(h)))
        self.h = h

    @classmethod
    def from_workload(cls, w, **kw):
        args = dict(n_layers=w.n_layers, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                    head_dim=w.head_dim, kv_dtype=w.kv_dtype, max_batch=w.batch,
                    max_tokens=w.max_tokens(), n_sink=w.n_sink, recent_window=w.recent_window,
                    budget_mode=w.budget_mode, budgets=w.budgets,
                    reclassify_interval=w.reclassify_interval, t2_scale_gran=w.t2_scale_gran,
                    t2_scale_dtype=w.t2_scale_dtype)
        args.update(kw)
        return cls(**args)

    # -------------------------------------------------------------- helpers
    def _check(self, status):
        L.check(status, self.h)

    def _enter(self):
        self.compute.wait_stream(torch.cuda.current_stream(self.device))

    def _leave(self, *tensors):
        cur = torch.cuda.current_stream(self.device)
        cur.wait_stream(self.compute)
        for t in tensors:
            t.record_stream(self.compute)

    def close(self):
        if getattr(self, "h", None):
            self._check(self.lib.tkv_destroy(self.h))
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---------------------------------------------------------------- API
    def append(self, seq: int, k: torch.Tensor, v: torch.Tensor, is_prompt: bool):
        """k, v: device tensors [L, n, Hkv, d] in the KV dtype."""
        k, v = k.contiguous(), v.contiguous()
        self._enter()
        self._check(self.lib.tkv_append(self.h, seq, _ptr(k), _ptr(v), k.shape[1], int(is_prompt)))
        self._leave(k, v)

    def decode_step(self, q, k_new, v_new, out=None):
        """q [B, L, Hq, d], k_new/v_new [B, L, Hkv, d] device tensors -> out [B, L, Hq, d]."""
        q, k_new, v_new = q.contiguous(), k_new.contiguous(), v_new.contiguous()
        if out is None:
            out = torch.empty_like(q)
        self._enter()
        self._check(self.lib.tkv_decode_step(self.h, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out)))
        self._leave(q, k_new, v_new, out)
        return out

    def decode_step_host(self, q, k_new, v_new, out=None):
        """The same step with host tensors (pinned for asynchronous copies)."""
        if out is None:
            out = torch.empty_like(q)
        self._check(self.lib.tkv_decode_step_host(self.h, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out)))
        return out

    def reclassify(self):
        self._enter()
        self._check(self.lib.tkv_reclassify(self.h))

    def prefetch(self, layer: int, slot: int):
        self._check(self.lib.tkv_prefetch(self.h, layer, slot))

    def synchronize(self):
        self._check(self.lib.tkv_synchronize(self.h))

    def test_stall_next_attention(self, wait_limit_ns: int):
        """Test hook: the next attention launch withholds one page copy, so a
        bounded device wait (limit wait_limit_ns) runs out; see tkv.h."""
        self._check(self.lib.tkv_test_stall_next_attention(self.h, int(wait_limit_ns)))

    def test_inject_fault(self, site: str, countdown: int = 1):
        """Test hook: the countdown-th visit of host call site `site` ("h2d",
        "d2h", "prefetch", "classify_overflow"; "none" disarms) is reported as
        failed; see tkv.h."""
        self._check(self.lib.tkv_test_inject_fault(self.h, L.FAULT_SITES[site], int(countdown)))

    def test_plant_bad_page(self, seq: int, tier: int, index: int) -> int:
        """Debug-build test hook: page-list entry `index` of (seq, tier) in the
        device table becomes the pool's capacity (one past its end); returns
        that id. See tkv.h."""
        planted = ctypes.c_int32()
        self._check(self.lib.tkv_test_plant_bad_page(self.h, seq, tier, index, ctypes.byref(planted)))
        return planted.value

    def num_sequences(self) -> int:
        n = ctypes.c_int32()
        self._check(self.lib.tkv_num_sequences(self.h, ctypes.byref(n)))
        return n.value

    def seq_len(self, seq: int) -> int:
        n = ctypes.c_int64()
        self._check(self.lib.tkv_seq_len(self.h, seq, ctypes.byref(n)))
        return n.value

    def scores(self, seq: int) -> np.ndarray:
        n = self.seq_len(seq)
        out = np.empty(n, dtype=np.float64)
        self._check(self.lib.tkv_get_scores(self.h, seq, out.ctypes.data, n))
        return out

    def set_scores(self, seq: int, s) -> None:
        s = np.ascontiguousarray(s, dtype=np.float64)
        self._enter()
        self._check(self.lib.tkv_set_scores(self.h, seq, s.ctypes.data, s.size))

    def tiers(self, seq: int) -> np.ndarray:
        n = self.seq_len(seq)
        out = np.empty(n, dtype=np.uint8)
        self._check(self.lib.tkv_get_tiers(self.h, seq, out.ctypes.data, n))
        return out

    def page_table(self, seq: int, tier: int):
        """(pages int32 [n], valid masks uint16 [n], positions int32 [n, 16]) of one tier."""
        n = ctypes.c_int64()
        self._check(self.lib.tkv_get_page_table(self.h, seq, tier, None, None, None, 0, ctypes.byref(n)))
        cap = n.value
        pages = np.empty(cap, dtype=np.int32)
        masks = np.empty(cap, dtype=np.uint16)
        pos = np.empty((cap, 16), dtype=np.int32)
        self._check(self.lib.tkv_get_page_table(self.h, seq, tier, pages.ctypes.data, masks.ctypes.data,
                                                pos.ctypes.data, cap, ctypes.byref(n)))
        return pages, masks, pos

    def t2_row(self, seq: int, pos: int):
        """(codes int8 [L, 2, Hkv, d], scales float32 [L, 2] or float16 [L, 2, Hkv])."""
        Ln, _, Hkv, d = self.shape
        codes = np.empty((Ln, 2, Hkv, d), dtype=np.int8)
        if self.t2_scale_gran == "token":
            scales = np.empty((Ln, 2), dtype=np.float32)
        else:
            scales = np.empty((Ln, 2, Hkv), dtype=np.float16)
        self._check(self.lib.tkv_get_t2_row(self.h, seq, pos, codes.ctypes.data, scales.ctypes.data))
        return codes, scales

    def kv_row(self, seq: int, pos: int):
        """Values a T0/T1 position holds: (k, v) float32 [L, Hkv, d]."""
        Ln, _, Hkv, d = self.shape
        k = torch.empty((Ln, Hkv, d), dtype=self.torch_dtype)
        v = torch.empty_like(k)
        self._check(self.lib.tkv_get_kv_row(self.h, seq, pos, _ptr(k), _ptr(v)))
        return k.float(), v.float()

    def stats(self) -> dict:
        st = L.Stats()
        self._check(self.lib.tkv_get_stats(self.h, ctypes.byref(st)))
        d = {name: getattr(st, name) for name, _ in L.Stats._fields_}
        d["tier_counts"] = list(st.tier_counts)
        return d

    def reset_stats(self):
        self._check(self.lib.tkv_reset_stats(self.h))


def inject_create_fault(countdown: int = 1):
    """Test hook: the countdown-th set-up call of the next tkv_create is
    reported as failed (0 disarms); see tkv.h."""
    lib = L.load()
    if countdown == 0:
        L.check(lib.tkv_test_inject_fault(None, 0, 0))
    else:
        L.check(lib.tkv_test_inject_fault(None, L.FAULT_SITES["alloc"], int(countdown)))


# ------------------------------------------------------------ stateless calls
def paged_attention(q, pool, page_table, slot_mask, page_counts, out=None, alpha_sum=None,
                    scratch=None, stream=None):
    """Split-K decode attention over one page pool (see tkv_paged_attention).

    q [B, Hq, d]; pool [pages, Hkv, 2, 16, d]; page_table int32 [B, max_pages];
    slot_mask int32/uint32 [pages]; page_counts host ints [B];
    alpha_sum float32 [B, Hkv, max_pages * 16] or None (accumulated into).
    """
    lib = L.load()
    B, Hq, d = q.shape
    Hkv = pool.shape[1]
    max_pages = page_table.shape[1]
    dt = L.DTYPE_BF16 if q.dtype == torch.bfloat16 else L.DTYPE_F32
    need = ctypes.c_size_t()
    L.check(lib.tkv_paged_attention_scratch_size(B, Hq, Hkv, d, max_pages, ctypes.byref(need)))
    if scratch is None:
        scratch = torch.empty(need.value, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    counts = np.ascontiguousarray(page_counts, dtype=np.int32)
    st = stream if stream is not None else torch.cuda.current_stream(q.device)
    L.check(lib.tkv_paged_attention(B, Hq, Hkv, d, dt, _ptr(q), _ptr(pool), _ptr(page_table),
                                    _ptr(slot_mask), counts.ctypes.data, max_pages, _ptr(out),
                                    _ptr(alpha_sum) if alpha_sum is not None else None,
                                    _ptr(scratch), scratch.numel(), st.cuda_stream))
    return out


def classify(scores, old_tier, params, n_sink, recent_window, stream=None):
    """Tier reassignment for B sequences (see tkv_classify). params: int64 [B, 5]."""
    lib = L.load()
    B, stride = scores.shape
    need = ctypes.c_size_t()
    L.check(lib.tkv_classify_scratch_size(B, stride, ctypes.byref(need)))
    scratch = torch.empty(need.value, dtype=torch.uint8, device=scores.device)
    new = torch.empty_like(old_tier)
    prm = np.ascontiguousarray(params, dtype=np.int64)
    st = stream if stream is not None else torch.cuda.current_stream(scores.device)
    L.check(lib.tkv_classify(B, _ptr(scores), _ptr(old_tier), _ptr(new), stride, prm.ctypes.data,
                             n_sink, recent_window, _ptr(scratch), scratch.numel(), st.cuda_stream))
    return new


def quantize_rows(x, scale_dtype="f32", stream=None):
    """8-bit absmax codes of the rows of x [rows, row_len] (see tkv_quantize_rows)."""
    lib = L.load()
    rows, n = x.shape
    dt = L.DTYPE_BF16 if x.dtype == torch.bfloat16 else L.DTYPE_F32
    codes = torch.empty((rows, n), dtype=torch.int8, device=x.device)
    scales = torch.empty(rows, dtype=torch.float32 if scale_dtype == "f32" else torch.float16, device=x.device)
    st = stream if stream is not None else torch.cuda.current_stream(x.device)
    L.check(lib.tkv_quantize_rows(_ptr(x), dt, rows, n, _ptr(codes), _ptr(scales),
                                  L.SCALE_F32 if scale_dtype == "f32" else L.SCALE_F16, st.cuda_stream))
    return codes, scales
