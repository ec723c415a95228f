"""8-bit storage of T2 tokens, specified in float32.

Methodology 1 and Results 4 ("Not All Thoughts Need HBM"): T2 keeps low-
importance tokens at reduced precision, for example 8-bit quantisation, and
those tokens are still read (the page reports an accuracy change from 8-bit T2
that differs from eviction).

Reading (the page names no scheme): symmetric absmax quantisation. For a row x
(one layer, one token, K or V, over all KV heads — or over one head when the
scale is per token and head):
    scale = absmax(x) / 127                (IEEE float32 division, rounded to
                                            nearest; then to float16 when the
                                            scale is stored as float16)
    code  = clamp(round_half_even(x / scale_used), -127, 127)  (float32 divide)
    absmax = 0 gives scale 0 and all codes 0.
Dequantisation is code * scale, exact in float64. A token promoted out of T2
keeps the lossy value: storage_dtype(float32(code * scale)).
This step is written in float32 on purpose so that codes can be compared bit
for bit. Pins: the absmax element maps to +-127, |x - dequant| <= scale / 2,
the all-zero row, and hand-worked vectors.
"""
from __future__ import annotations

import numpy as np


def quantize_rows(x, scale_dtype: str = "f32"):
    """x: float32 [..., m]. Returns (codes int8 [..., m], scale [...]) where the
    scale is float32, or float16 when scale_dtype == "f16"."""
    x = np.asarray(x, dtype=np.float32)
    absmax = np.max(np.abs(x), axis=-1)
    scale32 = (absmax / np.float32(127.0)).astype(np.float32)
    if scale_dtype == "f16":
        stored = scale32.astype(np.float16)
        divisor = stored.astype(np.float32)
    else:
        stored = scale32
        divisor = scale32
    div = divisor[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = (x / div).astype(np.float32)
    codes = np.where(div > 0, np.clip(np.rint(ratio), -127, 127), 0).astype(np.int8)
    return codes, stored


def dequantize(codes, scale) -> np.ndarray:
    """code * scale in float64 (exact: an int8 times a float32 or float16)."""
    s = np.asarray(scale).astype(np.float64)
    return np.asarray(codes).astype(np.float64) * s[..., None]


def bf16_round(x32: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16, ties to even (as float32)."""
    b = np.asarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> 16) & 1
    r = ((b + 0x7FFF + lsb) >> 16) << 16
    return (r & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def to_storage(codes, scale, kv_dtype: str) -> np.ndarray:
    """Value a token carries after promotion out of T2 (returned as float64)."""
    s = np.asarray(scale).astype(np.float32)
    prod = (np.asarray(codes).astype(np.float32) * s[..., None]).astype(np.float32)
    if kv_dtype == "bf16":
        prod = bf16_round(prod)
    return prod.astype(np.float64)
