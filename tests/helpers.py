"""Shared plumbing of the parity tests: prefill both sides from the seeded
generator, and regenerate slices for sampled full-size checks."""
from __future__ import annotations

import numpy as np
from oracle import decode_attention, quantize_rows
from oracle.quant import dequantize

SCORE_RTOL, SCORE_ATOL = 1e-4, 1e-7   # spec score tolerance (+ floor for fp32 underflow)
OUT_ATOL = 2e-2                        # attention output tolerance (bf16 I/O, fp32 accumulate)


def prefill_cache(cache, w, device, batches=None):
    """Append each request's seeded context: the prompt part, then the rest."""
    for b in (range(w.batch) if batches is None else batches):
        n, P = w.context_lens()[b], w.prompt_lens()[b]
        for lo, hi, prompt in ((0, P, True), (P, n, False)):
            if hi > lo:
                cache.append(b, w.kv_layers("k", b, lo, hi, device), w.kv_layers("v", b, lo, hi, device), prompt)


def prefill_oracle(oc, w, values=True):
    for b in range(w.batch):
        n, P = w.context_lens()[b], w.prompt_lens()[b]
        for lo, hi, prompt in ((0, P, True), (P, n, False)):
            if hi > lo:
                if values:
                    oc.append(b, w.kv_layers("k", b, lo, hi).float().numpy(), w.kv_layers("v", b, lo, hi).float().numpy(), prompt)
                else:
                    oc.append(b, None, None, prompt, n=hi - lo)


def assert_scores_close(got, want, what=""):
    got, want = np.asarray(got), np.asarray(want)
    bad = np.abs(got - want) > SCORE_RTOL * np.abs(want) + SCORE_ATOL
    if bad.any():
        i = int(np.nonzero(bad)[0][0])
        raise AssertionError(f"{what}: {int(bad.sum())} scores differ; first at {i}: {got[i]} vs {want[i]}")


def assert_page_tables_equal(cache, oc, b, what=""):
    for t in range(3):
        pages, masks, pos = cache.page_table(b, t)
        table = oc.page_table(b, t)
        assert pages.tolist() == [p for p, _ in table], f"{what}: tier {t} page ids of request {b}"
        assert pos.tolist() == [s for _, s in table], f"{what}: tier {t} slot positions of request {b}"
        want_masks = [sum(1 << j for j, x in enumerate(s) if x >= 0) for _, s in table]
        assert masks.tolist() == want_masks, f"{what}: tier {t} valid masks of request {b}"


def oracle_t2_codes(w, b, pos):
    """Oracle codes/scales of one position, quantised from its full-precision row."""
    ks = np.stack([w.kv("k", b, l, pos, pos + 1)[:, 0].float().numpy() for l in range(w.n_layers)])
    vs = np.stack([w.kv("v", b, l, pos, pos + 1)[:, 0].float().numpy() for l in range(w.n_layers)])
    out = []
    for x in (ks, vs):  # [L, Hkv, d]
        if w.t2_scale_gran == "token":
            c, s = quantize_rows(x.reshape(w.n_layers, -1), w.t2_scale_dtype)
            out.append((c.reshape(x.shape), s))
        else:
            c, s = quantize_rows(x, w.t2_scale_dtype)
            out.append((c, s))
    return out


def layer_attention(w, b, layer, q_bl, tiers, n_total, gen_device="cpu"):
    """Oracle outputs [Hq, d] and alphas [Hq, |R|] of all heads of one (request,
    layer) over the retained set, T2 rows dequantised from the oracle's codes
    (valid while no token has been promoted out of T2). The seeded inputs may be
    regenerated on a CUDA device (bit-identical to the CPU generator) and are
    brought back to the CPU before any oracle arithmetic."""
    K = w.kv("k", b, layer, 0, n_total, gen_device).cpu().float().numpy().astype(np.float64).transpose(1, 0, 2)
    V = w.kv("v", b, layer, 0, n_total, gen_device).cpu().float().numpy().astype(np.float64).transpose(1, 0, 2)
    t2 = np.nonzero(tiers == 2)[0]
    if t2.size:
        for X in (K, V):
            rows = X[t2].astype(np.float32)               # [n2, Hkv, d]
            if w.t2_scale_gran == "token":
                c, s = quantize_rows(rows.reshape(len(t2), -1), w.t2_scale_dtype)
                X[t2] = dequantize(c, s).reshape(rows.shape)
            else:
                c, s = quantize_rows(rows, w.t2_scale_dtype)
                X[t2] = dequantize(c, s)
    R = np.nonzero(tiers != 3)[0]
    out, alpha = decode_attention(np.asarray(q_bl, dtype=np.float64), K[R], V[R])
    return out, alpha, R
