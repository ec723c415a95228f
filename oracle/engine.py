"""The whole decode-step loop over the four-tier cache, as plain state changes.

Per step t (steps count from 1), following "Not All Thoughts Need HBM":
  1. every request appends its new token at position N with tier T0 and
     score 0 (Methodology 1: the recent window lives in T0);
  2. for every layer and query head, attention of the new token over the
     retained set R = T0 u T1 u T2 (T2 read dequantised; T3 absent) —
     Methodology 3 and Results 4;
  3. s_i += (1/L) sum_l (1/H) sum_h alpha_{l,h}[i] over R (Methodology 2);
  4. if t is a multiple of Delta, reassign the tiers (Methodology 1 and 4) and
     carry out the data movement as state changes: allocator slots, T2 codes,
     and the value each token now holds.

Values are held in float64 exactly as each tier stores them: the bf16 or f32
input for T0/T1, code * scale for T2, and storage(float32(code * scale)) for a
token promoted out of T2 (full precision is gone once a token was quantised).
Pins: a hand-worked one-layer, two-head, two-step fixture (the new token is
appended before attention and attended by its own query; scores accumulate the
head-averaged weights), the increments of a step summing to 1, Proposition 1
(a T0/T1 split changes outputs by at most 1e-12), and tier / page-table
invariants over whole runs.
"""
from __future__ import annotations

import numpy as np

from .allocator import PagedAllocator
from .attention import decode_attention
from .classify import T0, T1, T2, T3, budgets_for, classify
from .quant import dequantize, quantize_rows, to_storage
from .scores import score_increment


class _Seq:
    def __init__(self, L, Hkv, d):
        self.N = 0
        self.prompt_len = 0
        self.tier = np.zeros(0, dtype=np.uint8)
        self.s = np.zeros(0, dtype=np.float64)
        self.K = np.zeros((L, 0, Hkv, d), dtype=np.float64)
        self.V = np.zeros((L, 0, Hkv, d), dtype=np.float64)
        self.codes: dict[int, tuple] = {}      # pos -> (kcodes, kscale, vcodes, vscale)

    def grow(self, k, v, n=None):
        if k is None:
            self.tier = np.concatenate([self.tier, np.zeros(n, dtype=np.uint8)])
            self.s = np.concatenate([self.s, np.zeros(n, dtype=np.float64)])
            self.N += n
            return
        n = k.shape[1]
        self.K = np.concatenate([self.K, np.asarray(k, dtype=np.float64)], axis=1)
        self.V = np.concatenate([self.V, np.asarray(v, dtype=np.float64)], axis=1)
        self.tier = np.concatenate([self.tier, np.zeros(n, dtype=np.uint8)])
        self.s = np.concatenate([self.s, np.zeros(n, dtype=np.float64)])
        self.N += n


class OracleCache:
    def __init__(self, n_layers, n_q_heads, n_kv_heads, head_dim, kv_dtype="bf16",
                 n_sink=4, recent_window=128, budget_mode="percent",
                 budgets=(50, 30, 10, 10), reclassify_interval=64,
                 t2_scale_gran="token", t2_scale_dtype="f32", t2_mode="attend",
                 page_size=16, track_values=True):
        self.L, self.Hq, self.Hkv, self.d = n_layers, n_q_heads, n_kv_heads, head_dim
        self.kv_dtype = kv_dtype
        self.n_sink, self.W = n_sink, recent_window
        self.budget_mode, self.budgets = budget_mode, tuple(budgets)
        self.delta = reclassify_interval
        self.t2_gran, self.t2_sdt, self.t2_mode = t2_scale_gran, t2_scale_dtype, t2_mode
        self.seqs: list[_Seq] = []
        self.alloc = [PagedAllocator(page_size) for _ in range(3)]
        self.t = 0
        # track_values=False keeps only tiers, scores and slots (for caches too
        # large to hold in float64); decode_step then needs values and refuses.
        self.track_values = track_values

    @classmethod
    def from_workload(cls, w, **kw):
        return cls(w.n_layers, w.n_q_heads, w.n_kv_heads, w.head_dim, w.kv_dtype,
                   w.n_sink, w.recent_window, w.budget_mode, w.budgets,
                   w.reclassify_interval, w.t2_scale_gran, w.t2_scale_dtype, **kw)

    # ------------------------------------------------------------- appends
    def append(self, b: int, k, v, is_prompt: bool, n: int | None = None) -> None:
        """k, v: [L, n, Hkv, d] values of n new positions of request b (T0, s = 0);
        without value tracking pass k = v = None and the count n."""
        if b == len(self.seqs):
            self.seqs.append(_Seq(self.L, self.Hkv, self.d))
        sq = self.seqs[b]
        p0 = sq.N
        if self.track_values:
            sq.grow(np.asarray(k), np.asarray(v))
        else:
            sq.grow(None, None, n if n is not None else k.shape[1])
        if is_prompt:
            if p0 != sq.prompt_len:
                raise ValueError("prompt tokens must come before generated ones")
            sq.prompt_len += sq.N - p0
        self.alloc[T0].place(b, range(p0, sq.N))

    # ---------------------------------------------------------- the step
    def retained(self, b: int) -> np.ndarray:
        t = self.seqs[b].tier
        keep = t != T3
        if self.t2_mode == "mask":
            keep &= t != T2
        return np.nonzero(keep)[0]

    def attend(self, b: int, layer: int, q) -> tuple[np.ndarray, np.ndarray]:
        """Attention of query q [Hq, d] over request b's retained set at a layer."""
        sq = self.seqs[b]
        R = self.retained(b)
        out, alpha = decode_attention(q, sq.K[layer, R], sq.V[layer, R])
        return out, alpha

    def decode_step(self, q, k_new, v_new):
        """q: [B, L, Hq, d]; k_new, v_new: [B, L, Hkv, d].

        Returns (out [B, L, Hq, d] float64, [(R_b, delta_s_b)] per request)."""
        if not self.track_values:
            raise RuntimeError("decode_step needs value tracking")
        q = np.asarray(q, dtype=np.float64)
        B = q.shape[0]
        for b in range(B):
            self.append(b, np.asarray(k_new)[b][:, None], np.asarray(v_new)[b][:, None],
                        is_prompt=False)
        out = np.zeros((B, self.L, self.Hq, self.d), dtype=np.float64)
        deltas = []
        for b in range(B):
            R = self.retained(b)
            alphas = []
            for layer in range(self.L):
                out[b, layer], a = self.attend(b, layer, q[b, layer])
                alphas.append(a)
            ds = score_increment(alphas)
            self.seqs[b].s[R] += ds
            deltas.append((R, ds))
        self.t += 1
        if self.t % self.delta == 0:
            self.reclassify()
        return out, deltas

    # ------------------------------------------------------- reassignment
    def new_tiers(self, b: int) -> np.ndarray:
        sq = self.seqs[b]
        n0, n1, n2 = budgets_for(sq.N, self.budget_mode, self.budgets)
        return classify(sq.s, sq.tier, sq.prompt_len, self.n_sink, self.W, n0, n1, n2)

    def reclassify(self) -> None:
        for b, sq in enumerate(self.seqs):
            new = self.new_tiers(b)
            old = sq.tier
            moved = np.nonzero(new != old)[0]
            if self.track_values:
                for pos in moved:
                    self._move_values(sq, int(pos), int(old[pos]), int(new[pos]))
            for x in (T0, T1, T2):
                self.alloc[x].vacate(b, [p for p in moved if old[p] == x])
            for x in (T0, T1, T2):
                self.alloc[x].place(b, [p for p in moved if new[p] == x])
            # T0 lives in HBM: repack it so attention reads no empty slots (the
            # moves stay on the device; values are position-indexed here)
            self.alloc[T0].compact(b)
            sq.tier = new

    def _move_values(self, sq: _Seq, pos: int, src: int, dst: int) -> None:
        if dst == T3:
            sq.codes.pop(pos, None)
            return
        if dst == T2 and src != T2:
            kc, ks = self._quantize(sq.K[:, pos])
            vc, vs = self._quantize(sq.V[:, pos])
            sq.codes[pos] = (kc, ks, vc, vs)
            sq.K[:, pos] = self._dequantize(kc, ks)
            sq.V[:, pos] = self._dequantize(vc, vs)
        elif src == T2 and dst != T2:
            kc, ks, vc, vs = sq.codes.pop(pos)
            sq.K[:, pos] = self._promote(kc, ks)
            sq.V[:, pos] = self._promote(vc, vs)

    def _quantize(self, x):
        """x: [L, Hkv, d] float64 holding float32-exact values."""
        x32 = np.asarray(x, dtype=np.float32)
        if self.t2_gran == "token":
            codes, scale = quantize_rows(x32.reshape(self.L, -1), self.t2_sdt)
            return codes.reshape(x32.shape), scale                  # scale [L]
        codes, scale = quantize_rows(x32, self.t2_sdt)              # scale [L, Hkv]
        return codes, scale

    def _dequantize(self, codes, scale):
        if self.t2_gran == "token":
            return dequantize(codes.reshape(self.L, -1), scale).reshape(codes.shape)
        return dequantize(codes, scale)

    def _promote(self, codes, scale):
        if self.t2_gran == "token":
            v = to_storage(codes.reshape(self.L, -1), scale, self.kv_dtype)
            return v.reshape(codes.shape)
        return to_storage(codes, scale, self.kv_dtype)

    # ------------------------------------------------------ introspection
    def set_scores(self, b: int, s) -> None:
        s = np.asarray(s, dtype=np.float64)
        if np.isnan(s).any():
            raise ValueError("NaN score")
        self.seqs[b].s = s.copy()

    def page_table(self, b: int, tier: int):
        return self.alloc[tier].table(b)
