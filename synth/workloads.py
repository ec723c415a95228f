"""The five synthetic workloads of the tiered decode step, and their inputs.

Every tensor here is a pure function of the workload's seed and of indices, so
the oracle (CPU) and the CUDA path (device) see the same bits. Nothing in this
file computes attention, scores, tiers or quantisation: it only makes inputs.

Shapes follow the decode-step problem of "Not All Thoughts Need HBM":
L layers, Hq query heads, Hkv key/value heads, head dimension d.

Streams (the fourth Philox counter word) keep the inputs independent:
K, V, Q, per-position key scale, context lengths, spike positions, spike
directions and synthetic score vectors.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field
from functools import lru_cache

import torch

from .philox import normal_f32, uniform_u32

S_K, S_V, S_Q, S_KSCALE, S_CTX, S_SPIKE, S_DIR, S_SCORE = 1, 2, 3, 4, 5, 6, 7, 8

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    kv_dtype: str                 # "f32" | "bf16"
    batch: int
    n_sink: int
    recent_window: int
    budget_mode: str              # "percent" | "count"
    budgets: tuple                # (t0, t1, t2, t3): integer percents, or counts
    reclassify_interval: int      # Delta
    context: tuple                # ("fixed", n) | ("uniform", lo, hi)
    prompt_len: int = 0
    key_scale: tuple = ("none",)  # ("lognormal", sigma) | ("spikes", count, factor)
                                  # | ("delayed_spikes", fraction, factor, delay, groups)
    t2_scale_gran: str = "token"  # "token" | "token_head"
    t2_scale_dtype: str = "f32"   # "f32" | "f16"
    n_steps: int = 16
    seed: int = 0
    page_size: int = 16

    # ----------------------------------------------------------------- shape
    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def torch_dtype(self):
        return DTYPES[self.kv_dtype]

    @property
    def elem_bytes(self) -> int:
        return 4 if self.kv_dtype == "f32" else 2

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    # ------------------------------------------------------------ per request
    def context_lens(self) -> list[int]:
        kind = self.context[0]
        if kind == "fixed":
            return [int(self.context[1])] * self.batch
        lo, hi = int(self.context[1]), int(self.context[2])
        u = uniform_u32(self.seed, S_CTX, 0, 0, 0, self.batch)
        return [lo + int((int(x) * (hi - lo + 1)) >> 32) for x in u]

    def prompt_lens(self) -> list[int]:
        return [min(self.prompt_len, n) for n in self.context_lens()]

    def max_tokens(self) -> int:
        return max(self.context_lens()) + self.n_steps

    def total_len(self, b: int) -> int:
        return self.context_lens()[b] + self.n_steps

    # -------------------------------------------------------------- key scale
    def spike_positions(self, b: int) -> torch.Tensor:
        """Sorted positions whose keys carry a spike (empty if none)."""
        return _spike_positions(self, b)

    def key_scales(self, b: int) -> torch.Tensor:
        """float32 [total_len(b)]: per-position multiplier of the key noise."""
        return _key_scales(self, b)

    def spike_vectors(self, layer: int, kvh: int) -> torch.Tensor:
        """float32 [groups, d]: the spike offset added to a spike key of each group."""
        return _spike_vectors(self, layer, kvh)

    def spike_groups(self, b: int) -> tuple[torch.Tensor, torch.Tensor]:
        """(group of each spike position, first position of each group)."""
        pos = self.spike_positions(b)
        g = int(self.key_scale[4])
        if pos.numel() == 0:
            return torch.zeros(0, dtype=torch.int64), torch.zeros(0, dtype=torch.int64)
        grp = (torch.arange(pos.numel()) * g) // pos.numel()
        first = torch.stack([pos[grp == j].min() for j in range(g)])
        return grp, first

    # ------------------------------------------------------------------ K / V
    def kv(self, which: str, b: int, layer: int, pos0: int, pos1: int,
           device="cpu") -> torch.Tensor:
        """Keys or values of positions [pos0, pos1) of request b at one layer.

        Returns [Hkv, pos1 - pos0, d] in the workload's storage dtype. A key is
        round(z * scale[pos] (+ spike offset)), a value is round(z); z ~ N(0, 1).
        """
        d, hk = self.head_dim, self.n_kv_heads
        n = pos1 - pos0
        stream = S_K if which == "k" else S_V
        a = (b << 16) | layer
        heads = torch.arange(hk, dtype=torch.int64)
        z = normal_f32(self.seed, stream, a, heads, pos0 * d, n * d, device)
        z = z.reshape(hk, n, d)
        if which == "k":
            sc = self.key_scales(b)[pos0:pos1].to(device)
            z = z * sc.view(1, n, 1)
            if self.key_scale[0] == "delayed_spikes":
                pos = self.spike_positions(b)
                grp, _ = self.spike_groups(b)
                sel = (pos >= pos0) & (pos < pos1)
                if bool(sel.any()):
                    p_local = (pos[sel] - pos0).to(device)
                    g_sel = grp[sel]
                    for h in range(hk):
                        sv = self.spike_vectors(layer, h).to(device)
                        z[h, p_local] = z[h, p_local] + sv[g_sel.to(device)]
        return z.to(self.torch_dtype)

    def kv_layers(self, which: str, b: int, pos0: int, pos1: int,
                  device="cpu") -> torch.Tensor:
        """[L, pos1 - pos0, Hkv, d]: the prefill layout the library takes."""
        out = torch.empty(self.n_layers, pos1 - pos0, self.n_kv_heads, self.head_dim,
                          dtype=self.torch_dtype, device=device)
        for layer in range(self.n_layers):
            out[layer] = self.kv(which, b, layer, pos0, pos1, device).permute(1, 0, 2)
        return out

    def step_positions(self, step: int) -> list[int]:
        """Position of the token decoded at step `step` (steps count from 1)."""
        return [n + step - 1 for n in self.context_lens()]

    def kv_new(self, which: str, step: int, device="cpu") -> torch.Tensor:
        """[B, L, Hkv, d]: the key or value appended at decode step `step`."""
        d, hk, L = self.head_dim, self.n_kv_heads, self.n_layers
        out = torch.empty(self.batch, L, hk, d, dtype=self.torch_dtype, device=device)
        stream = S_K if which == "k" else S_V
        layers = torch.arange(L, dtype=torch.int64).view(L, 1)
        heads = torch.arange(hk, dtype=torch.int64).view(1, hk)
        for b, p in enumerate(self.step_positions(step)):
            if which == "k" and self.key_scale[0] == "delayed_spikes":
                for layer in range(L):
                    out[b, layer] = self.kv(which, b, layer, p, p + 1, device)[:, 0, :]
                continue
            z = normal_f32(self.seed, stream, (b << 16) | layers, heads, p * d, d, device)  # [L, Hkv, d]
            if which == "k":
                z = z * self.key_scales(b)[p].to(device)
            out[b] = z.to(self.torch_dtype)
        return out

    # --------------------------------------------------------------- queries
    def queries(self, step: int, device="cpu") -> torch.Tensor:
        """[B, L, Hq, d]: the queries of decode step `step` (from 1)."""
        B, L, H, d = self.batch, self.n_layers, self.n_q_heads, self.head_dim
        if self.key_scale[0] == "delayed_spikes":
            z = normal_f32(self.seed, S_Q, step, 0, 0, B * L * H * d, "cpu").reshape(B, L, H, d)
            return _delayed_spike_queries(self, step, z).to(self.torch_dtype).to(device)
        z = normal_f32(self.seed, S_Q, step, 0, 0, B * L * H * d, device).reshape(B, L, H, d)
        return z.to(self.torch_dtype)

    # ----------------------------------------------------------------- scores
    def synthetic_scores(self, b: int, n: int, ties: bool = True) -> torch.Tensor:
        """float64 [n] non-negative scores; with ties=True many values repeat."""
        u = uniform_u32(self.seed, S_SCORE, b, 0, 0, n)
        if ties:
            return ((u >> 22).to(torch.float64)) * (2.0 ** -10)
        return u.to(torch.float64) * (2.0 ** -32)


# ---------------------------------------------------------------- helpers
@lru_cache(maxsize=256)
def _spike_positions(w: Workload, b: int) -> torch.Tensor:
    kind = w.key_scale[0]
    if kind not in ("spikes", "delayed_spikes"):
        return torch.zeros(0, dtype=torch.int64)
    total = w.total_len(b)
    if kind == "spikes":
        lo, count = 0, int(w.key_scale[1])
        hi = w.context_lens()[b]
    else:
        lo, hi = w.prompt_lens()[b], total
        count = int(round(float(w.key_scale[1]) * total))
    count = min(count, hi - lo)
    u = uniform_u32(w.seed, S_SPIKE, b, 0, lo, hi - lo)
    key = u * (1 << 20) + torch.arange(hi - lo, dtype=torch.int64)  # ties by position
    order = torch.argsort(key)
    return torch.sort(order[:count] + lo).values


@lru_cache(maxsize=256)
def _key_scales(w: Workload, b: int) -> torch.Tensor:
    total = w.total_len(b)
    kind = w.key_scale[0]
    if kind == "lognormal":
        z = normal_f32(w.seed, S_KSCALE, b, 0, 0, total).to(torch.float64)
        return torch.exp(float(w.key_scale[1]) * z).to(torch.float32)
    s = torch.ones(total, dtype=torch.float32)
    if kind == "spikes":
        s[_spike_positions(w, b)] = float(w.key_scale[2])
    return s


@lru_cache(maxsize=4096)
def _spike_dirs(w: Workload, layer: int, kvh: int) -> torch.Tensor:
    """float64 [groups, d] orthonormal directions for one (layer, kv head)."""
    g, d = int(w.key_scale[4]), w.head_dim
    z = normal_f32(w.seed, S_DIR, layer, kvh, 0, g * d).to(torch.float64).reshape(g, d)
    q, _ = torch.linalg.qr(z.T)
    return q.T.contiguous()


@lru_cache(maxsize=4096)
def _spike_vectors(w: Workload, layer: int, kvh: int) -> torch.Tensor:
    amp = float(w.key_scale[2]) * math.sqrt(w.head_dim)
    return (amp * _spike_dirs(w, layer, kvh)).to(torch.float32)


def _delayed_spike_queries(w: Workload, step: int, z: torch.Tensor) -> torch.Tensor:
    """q = P_perp g + sum of the directions of the groups active at this position."""
    delay = int(w.key_scale[3])
    out = torch.empty_like(z)
    G = w.group
    for b, p in enumerate(w.step_positions(step)):
        _, first = w.spike_groups(b)
        active = (first + delay) <= p
        for layer in range(w.n_layers):
            for kvh in range(w.n_kv_heads):
                e = _spike_dirs(w, layer, kvh)                      # [g, d] f64
                g = z[b, layer, kvh * G:(kvh + 1) * G].to(torch.float64)  # [G, d]
                g = g - (g @ e.T) @ e
                if bool(active.any()):
                    g = g + e[active].sum(0, keepdim=True)
                out[b, layer, kvh * G:(kvh + 1) * G] = g.to(torch.float32)
    return out


# ------------------------------------------------------------- the configs
TINY = Workload(
    name="tiny", n_layers=1, n_q_heads=8, n_kv_heads=2, head_dim=64, kv_dtype="f32",
    batch=1, n_sink=4, recent_window=64, budget_mode="count", budgets=(256, 128, 64, 0),
    reclassify_interval=4, context=("fixed", 512), prompt_len=32,
    key_scale=("spikes", 16, 4.0), n_steps=16, seed=11)

CHAIN7B = Workload(
    name="chain7b", n_layers=28, n_q_heads=28, n_kv_heads=4, head_dim=128, kv_dtype="bf16",
    batch=1, n_sink=4, recent_window=128, budget_mode="percent", budgets=(50, 30, 10, 10),
    reclassify_interval=32, context=("fixed", 256), prompt_len=256,
    key_scale=("lognormal", 0.5), n_steps=2000, seed=12)

BATCH32 = Workload(
    name="batch32", n_layers=28, n_q_heads=28, n_kv_heads=4, head_dim=128, kv_dtype="bf16",
    batch=32, n_sink=4, recent_window=128, budget_mode="percent", budgets=(40, 40, 10, 10),
    reclassify_interval=64, context=("uniform", 1024, 8192), prompt_len=0,
    key_scale=("lognormal", 0.5), n_steps=256, seed=13)

MHA16K = Workload(
    name="mha16k", n_layers=32, n_q_heads=32, n_kv_heads=32, head_dim=128, kv_dtype="bf16",
    batch=8, n_sink=4, recent_window=128, budget_mode="percent", budgets=(25, 50, 15, 10),
    reclassify_interval=64, context=("fixed", 15360), prompt_len=512,
    key_scale=("delayed_spikes", 0.01, 6.0, 500, 16), t2_scale_gran="token_head",
    t2_scale_dtype="f16", n_steps=1024, seed=14)


def long128k(t0: int) -> Workload:
    return Workload(
        name=f"long128k_t0_{t0}", n_layers=32, n_q_heads=32, n_kv_heads=8, head_dim=128,
        kv_dtype="bf16", batch=4, n_sink=4, recent_window=128, budget_mode="percent",
        budgets=(t0, 95 - t0, 0, 5), reclassify_interval=64, context=("fixed", 131072),
        prompt_len=0, key_scale=("lognormal", 1.0), n_steps=64, seed=15)


def batch32_budget(name: str, budgets: tuple) -> Workload:
    """The batch-32 serving shape under another tier budget (the pages'
    experimental axes, measured here as system cost): full cache, eviction
    without offload, and the share of HBM at fixed eviction."""
    return BATCH32.replace(name=name, budgets=budgets)


BUDGET_VARIANTS = [batch32_budget("batch32_full", (100, 0, 0, 0)),
                   batch32_budget("batch32_evict50", (50, 0, 0, 50)),
                   batch32_budget("batch32_hbm30", (30, 50, 10, 10)),
                   batch32_budget("batch32_hbm50", (50, 30, 10, 10)),
                   batch32_budget("batch32_hbm70", (70, 10, 10, 10))]

WORKLOADS = {w.name: w for w in (TINY, CHAIN7B, BATCH32, MHA16K,
                                 long128k(25), long128k(50), long128k(75), *BUDGET_VARIANTS)}
