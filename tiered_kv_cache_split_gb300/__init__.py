"""Tiered KV-cache decode step for GB300 (sm_103a).

The four-tier hierarchy of "Not All Thoughts Need HBM": T0 in HBM, T1 in
pinned host DDR prefetched before attention, T2 as 8-bit codes, T3 evicted;
importance is the cumulative attention score, reassigned every Delta steps.
All compute runs in the CUDA kernels of libtkv.so (C ABI: include/tkv.h);
this package only marshals arguments.
"""
from ._lib import TkvError, load
from .cache import TieredKVCache, classify, paged_attention, quantize_rows

__all__ = ["TieredKVCache", "TkvError", "load", "paged_attention", "classify", "quantize_rows"]
