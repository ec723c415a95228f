"""Counter-based uniform bits and standard normals, identical on CPU and CUDA.

The generator is Philox4x32-10 as published by Salmon, Moraes, Dror and Shaw,
"Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11): a 128-bit counter and a
64-bit key go through ten rounds, each of two 32x32->64 multiplies (constants
0xD2511F53 and 0xCD9E8D57) whose high halves are xored with the other counter
words and the round key; the key is bumped by the Weyl constants 0x9E3779B9 and
0xBB67AE85 between rounds.

Everything is written with int64 torch tensors whose values never exceed
2^63 - 1 (each 32-bit multiplier is split into 16-bit halves), so the same
Python code gives the same bits on a CPU tensor and on a CUDA tensor. That is
what lets the oracle regenerate any slice of a workload that the GPU generated
in bulk.

A standard normal is read from a 2^16-entry table of inverse-CDF values at the
midpoints (j + 1/2) / 2^16, evaluated once in float64 and rounded to float32,
indexed by 16 uniform bits. It is N(0, 1) quantised to 65,536 levels and cut at
about 4.3 sigma, which is plenty for bf16 test data.
"""
from __future__ import annotations

import statistics
from functools import lru_cache

import torch

MASK32 = 0xFFFFFFFF
_M0 = 0xD2511F53
_M1 = 0xCD9E8D57
_W0 = 0x9E3779B9
_W1 = 0xBB67AE85
ROUNDS = 10


def _mulhilo(a: torch.Tensor, m: int):
    """(hi, lo) 32-bit halves of a * m for 0 <= a, m < 2^32, without int64 overflow."""
    a0 = a & 0xFFFF
    a1 = a >> 16
    p0 = a0 * m                      # < 2^48
    p1 = a1 * m                      # < 2^48
    t = p1 + (p0 >> 16)              # a*m = t * 2^16 + (p0 & 0xFFFF)
    hi = t >> 16
    lo = ((t & 0xFFFF) << 16) | (p0 & 0xFFFF)
    return hi, lo


def philox4x32(c0, c1, c2, c3, k0: int, k1: int, rounds: int = ROUNDS):
    """Philox4x32-R on broadcastable int64 tensors holding 32-bit words.

    Returns the four 32-bit output words as int64 tensors.
    """
    k0 &= MASK32
    k1 &= MASK32
    for r in range(rounds):
        if r:
            k0 = (k0 + _W0) & MASK32
            k1 = (k1 + _W1) & MASK32
        hi0, lo0 = _mulhilo(c0, _M0)
        hi1, lo1 = _mulhilo(c2, _M1)
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


def _as_i64(x, device):
    if isinstance(x, torch.Tensor):
        return x.to(device=device, dtype=torch.int64)
    return torch.tensor(int(x), dtype=torch.int64, device=device)


def uniform_u16(seed: int, stream: int, a, b, start: int, count: int,
                device="cpu") -> torch.Tensor:
    """16-bit uniforms for elements [start, start + count) of stream (stream, a, b).

    Element i lives in Philox block i // 8 (counter = (i // 8, b, a, stream),
    key = the 64-bit seed); within a block, element 8c + 2w + h is the h-th
    16-bit half (low half first) of output word w. `a` and `b` may be int64
    tensors; they broadcast against a trailing element axis of length `count`.
    """
    if count == 0:
        shape = torch.broadcast_shapes(_as_i64(a, "cpu").shape, _as_i64(b, "cpu").shape)
        return torch.zeros(*shape, 0, dtype=torch.int64, device=device)
    first = start // 8
    last = (start + count - 1) // 8
    blk = torch.arange(first, last + 1, dtype=torch.int64, device=device)
    at = _as_i64(a, device).unsqueeze(-1) & MASK32
    bt = _as_i64(b, device).unsqueeze(-1) & MASK32
    c0 = blk & MASK32
    shape = torch.broadcast_shapes(c0.shape, at.shape, bt.shape)
    c0 = c0.expand(shape)
    c1 = bt.expand(shape)
    c2 = at.expand(shape)
    c3 = torch.full(shape, int(stream) & MASK32, dtype=torch.int64, device=device)
    w = philox4x32(c0, c1, c2, c3, seed & MASK32, (seed >> 32) & MASK32)
    words = torch.stack(w, dim=-1)                       # [..., nblk, 4]
    halves = torch.stack((words & 0xFFFF, words >> 16), dim=-1)  # [..., nblk, 4, 2]
    flat = halves.reshape(*shape[:-1], -1)               # [..., nblk * 8]
    off = start - first * 8
    return flat[..., off:off + count]


def uniform_u32(seed: int, stream: int, a, b, start: int, count: int,
                device="cpu") -> torch.Tensor:
    """32-bit uniforms: element i is the pair of 16-bit uniforms 2i, 2i + 1."""
    u = uniform_u16(seed, stream, a, b, 2 * start, 2 * count, device)
    u = u.reshape(*u.shape[:-1], count, 2)
    return u[..., 0] | (u[..., 1] << 16)


@lru_cache(maxsize=None)
def _normal_table_cpu() -> torch.Tensor:
    nd = statistics.NormalDist()
    vals = [nd.inv_cdf((j + 0.5) / 65536.0) for j in range(65536)]
    return torch.tensor(vals, dtype=torch.float64).to(torch.float32)


_TABLES: dict = {}


def normal_table(device="cpu") -> torch.Tensor:
    """The 65,536 float32 midpoint quantiles of N(0, 1), on `device`."""
    key = str(torch.device(device))
    t = _TABLES.get(key)
    if t is None:
        t = _normal_table_cpu().to(device)
        _TABLES[key] = t
    return t


def normal_f32(seed: int, stream: int, a, b, start: int, count: int,
               device="cpu") -> torch.Tensor:
    """Standard normals (float32) for elements [start, start + count) of a stream."""
    u = uniform_u16(seed, stream, a, b, start, count, device)
    return normal_table(device)[u]
