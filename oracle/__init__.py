"""CPU oracle for the tiered KV-cache decode step — TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 NumPy restatement of what one decode step over the
four-tier cache computes, following the summary page "Not All Thoughts Need
HBM" (arXiv 2605.09490). Citations in this package name that page's sections:

  * Problem statement                      (the ~800 MB per 2,000-token chain)
  * Methodology 1, four-tier classification (T0 HBM, T1 DDR, T2 8-bit, T3 evicted;
                                             protected prompt, sinks, recent window)
  * Methodology 2, importance scoring       (the cumulative-attention equation for s_i)
  * Methodology 3, zero-approximation-error offload (Proposition 1)
  * Methodology 4, system implementation    (reassignment every Delta = 64 steps,
                                             asynchronous differential prefetch)
  * Results 4, precision sensitivity        (T2 tokens are read at 8 bits)

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may import
this package. The library under tiered_kv_cache_split_gb300/ never does, and
shares no code, header, table or helper with it.

Parity status of each part (what pins it is listed in each module's header):
attention, scores, classifier, quantiser and allocator are pinned by tests;
end-to-end model accuracy is "parity unpinned" (it needs trained weights and
benchmark datasets that the pages only summarise).
"""
from .attention import decode_attention
from .classify import budgets_for, classify, protected_mask
from .quant import dequantize, quantize_rows, to_storage
from .scores import score_increment
from .allocator import PagedAllocator
from .engine import OracleCache

__all__ = ["decode_attention", "score_increment", "classify", "protected_mask",
           "budgets_for", "quantize_rows", "dequantize", "to_storage",
           "PagedAllocator", "OracleCache"]
