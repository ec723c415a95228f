"""Benchmark of the tiered KV-cache decode step on GB300.

One step = one decode step of every request through all layers: append the new
token to T0, prefetch T1 and T2 of each layer on the copy stream, split-K
attention over T0 + T1 + T2 with the cumulative score fused into the softmax
epilogue, the float64 score fold, and (every Delta steps) tier reassignment with
differential data movement. The default workload is the batch-32 serving case:
32 requests of 1k-8k tokens (uniform), 28 layers, 28 query / 4 KV heads,
d = 128, bf16, 16-token pages, budgets T0/T1/T2/T3 = 40/40/10/10, Delta = 64.

Prints one JSON line (rank 0). `--impl reference` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode steps/s (KV-read GB/s as fraction of HBM peak in roofline)"


NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e, nominal


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _traffic(workload):
    """DRAM read + write bytes per attention launch from the committed ncu
    capture, or None when there is none for this workload or the kernel source
    changed since it was taken."""
    import hashlib
    tp = os.path.join(ROOT, "profiles", "attention_traffic.json")
    if not os.path.exists(tp):
        return None
    rec = json.load(open(tp)).get(workload)
    if not rec:
        return None
    src = os.path.join(ROOT, "tiered_kv_cache_split_gb300", "csrc", "attention.cu")
    if hashlib.sha256(open(src, "rb").read()).hexdigest() != rec.get("attention_cu_sha256"):
        return None
    return rec["traffic_bytes_per_launch"]


def _workload(name):
    from synth import WORKLOADS
    return WORKLOADS[name]


def _config(w, n_ranks, args=None):
    lens = w.context_lens()
    c = {"workload": w.name, "batch": w.batch, "layers": w.n_layers, "q_heads": w.n_q_heads,
         "kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "kv_dtype": w.kv_dtype,
         "context_tokens": {"min": min(lens), "max": max(lens), "mean": sum(lens) / len(lens)},
         "budgets": list(w.budgets), "budget_mode": w.budget_mode, "delta": w.reclassify_interval,
         "page_size": 16, "parallelism": f"replicas x{n_ranks}",
         "l2": "inputs larger than L2: each step streams GBs of KV through the 129 MB L2"}
    if args is not None:
        c["host_tiers"] = args.host_tiers
        c["layers_per_launch"] = args.layers_per_launch or "auto"
    return c


# ------------------------------------------------------------------ clocks
class ClockSampler:
    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ dist
def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(ws, x, device):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def kernel_name(w):
    """The attention kernel the workload's shape selects."""
    if w.kv_dtype == "bf16" and w.group >= 2:
        return "attn_split_mma_kernel"
    return "attn_split_fma_kernel"


# ------------------------------------------------------------------ GPU arm
def run_gpu(args):
    import torch
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from tiered_kv_cache_split_gb300 import TieredKVCache

    w = _workload(args.workload)
    if args.layers:
        w = w.replace(n_layers=args.layers)   # a smaller case of the same kernels, for profiling
    delta = w.reclassify_interval
    K, W = args.steps, args.warmup
    # untimed prefix: reach the tiered steady state (first reassignment at step
    # Delta), then W warm-up steps, and align so the timed window ends on a
    # multiple of Delta: it then holds ceil(K / Delta) reassignments.
    untimed = math.ceil((delta + W + K) / delta) * delta - K
    e2e_untimed = math.ceil(K / delta) * delta - K   # the e2e window also ends on a multiple of Delta
    total_steps = untimed + K + e2e_untimed + K
    w = w.replace(n_steps=total_steps + 1)

    cache = TieredKVCache.from_workload(w, timing=True, split_pages=args.split_pages, host_tiers=args.host_tiers,
                                        layers_per_launch=args.layers_per_launch)
    t0 = time.time()
    for b in range(w.batch):
        n, P = w.context_lens()[b], w.prompt_lens()[b]
        for lo, hi, prompt in ((0, P, True), (P, n, False)):
            if hi > lo:
                cache.append(b, w.kv_layers("k", b, lo, hi, dev), w.kv_layers("v", b, lo, hi, dev), prompt)
    torch.cuda.synchronize()
    prefill_s = time.time() - t0

    def inputs(t):
        return w.queries(t, dev), w.kv_new("k", t, dev), w.kv_new("v", t, dev)

    out = None
    step = 0
    # the untimed prefix only has to reach the tiered steady state: it cycles a
    # few generated input sets instead of generating every step's inputs
    pool = [inputs(i + 1) for i in range(4)]
    for _ in range(untimed):
        step += 1
        q, k, v = pool[step % len(pool)]
        out = cache.decode_step(q, k, v, out)
    timed_inputs = [inputs(step + i + 1) for i in range(K)]
    torch.cuda.synchronize()
    launches_before = cache.stats()["kernel_launches"]   # library launches before the timed region
    cache.reset_stats()
    stream = cache.compute
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        _barrier(ws)
        torch.cuda.synchronize()
        ev0.record(stream)
        for i in range(K):
            q, k, v = timed_inputs[i]
            out = cache.decode_step(q, k, v, out)
        ev1.record(stream)
        cache.synchronize()
        torch.cuda.synchronize()
        _barrier(ws)
    step += K
    ms = ev0.elapsed_time(ev1)
    st = cache.stats()
    ms_max = _max_over_ranks(ws, ms, dev)
    del timed_inputs

    # ---- end to end through the host-buffer entry point (pinned host in and out)
    for _ in range(e2e_untimed):
        step += 1
        q, k, v = pool[step % len(pool)]
        out = cache.decode_step(q, k, v, out)
    del pool
    host = []
    for i in range(K):
        q, k, v = inputs(step + i + 1)
        host.append((q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory()))
    out_h = torch.empty_like(host[0][0]).pin_memory()
    cache.synchronize()
    _barrier(ws)
    t0 = time.perf_counter()
    for i in range(K):
        q, k, v = host[i]
        cache.decode_step_host(q, k, v, out_h)
    cache.synchronize()
    e2e_s = time.perf_counter() - t0
    _barrier(ws)
    e2e_s = _max_over_ranks(ws, e2e_s, dev)
    h2d = sum(x.numel() * x.element_size() for x in host[0])
    d2h = out_h.numel() * out_h.element_size()

    # ---- host link probe: a plain pinned host -> device copy
    probe_h = torch.empty(2 << 30, dtype=torch.uint8).pin_memory()
    probe_d = torch.empty_like(probe_h, device=dev)
    probe_d.copy_(probe_h, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = 1e30
    for _ in range(3):
        e0.record()
        probe_d.copy_(probe_h, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    link_gbs = probe_h.numel() / best / 1e6
    # the same copy from the cache's own pinned workspace (the T1 pool is its
    # first region): tells a slow source buffer from a slow step pattern
    pool_view = cache._pin[:min(cache._pin.numel(), 151 << 20)]
    best_pool = 1e30
    for _ in range(3):
        e0.record()
        probe_d[:pool_view.numel()].copy_(pool_view, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        best_pool = min(best_pool, e0.elapsed_time(e1))
    pool_link_gbs = pool_view.numel() / best_pool / 1e6
    del probe_h, probe_d

    peak, peak_kind = _peaks()
    attn_ms = st["attn_ms"] / max(st["attn_launches"], 1)
    combine_ms = st["combine_ms"] / max(st["attn_launches"], 1)   # once per step, spread over the step's launches
    layers_per_launch = st["attn_layers"] / max(st["attn_launches"], 1)
    bytes_per_launch = st["attn_bytes"] / max(st["attn_launches"], 1)
    achieved = bytes_per_launch / (attn_ms * 1e6) if attn_ms > 0 else 0.0
    pair = bytes_per_launch / ((attn_ms + combine_ms) * 1e6) if attn_ms > 0 else 0.0
    prefetch_gbs = st["prefetch_bytes"] / (st["prefetch_ms"] * 1e6) if st["prefetch_ms"] > 0 else None
    launches = st["kernel_launches"]   # counted by the library over the timed region
    span_us = 1000.0 * st["attn_span_ms"] / max(st["attn_launches"], 1) if st["attn_span_ms"] > 0 else None
    span_gbs = bytes_per_launch / (span_us * 1e3) if span_us else None
    clocks = clk.summary()
    traffic = _traffic(w.name)
    line = {
        "metric": METRIC, "value": ws * K / (ms_max / 1000.0), "unit": "steps/s", "n_gpus": ws,
        "steps": K, "warmup": W, "ms_per_step": ms_max / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.kv_dtype, "data": "synthetic",
        "config": _config(w, ws, args),
        "roofline": {"bound": "hbm", "kernel": kernel_name(w), "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "frac_of_nominal": achieved / NOMINAL_HBM_GBS, "nominal_peak": NOMINAL_HBM_GBS,
                     "traffic": traffic, "bytes_per_launch": bytes_per_launch,
                     "layers_per_launch": layers_per_launch,
                     "bytes_per_layer": bytes_per_launch / max(layers_per_launch, 1),
                     "launch_ms": attn_ms, "combine_ms_per_launch": combine_ms,
                     "with_combine": {"achieved": pair, "frac": pair / peak},
                     # the kernel body alone: first CTA start to last CTA end (%globaltimer),
                     # without the launch and event overhead the CUDA-event figure includes
                     "device_span": {"us_per_launch": span_us, "achieved": span_gbs,
                                     "frac": span_gbs / peak if span_gbs else None}},
        "kv_read_gbs": achieved,
        "link": {"prefetch_gbs": prefetch_gbs, "probe_h2d_gbs": link_gbs, "probe_pool_h2d_gbs": pool_link_gbs,
                 "frac": (prefetch_gbs / link_gbs) if prefetch_gbs else None,
                 "prefetch_bytes_per_step": st["prefetch_bytes"] / K},
        "reclassify_ms": st["reclassify_ms"] / max(st["reclassifies"], 1) if st["reclassifies"] else None,
        "reclassify_breakdown_ms": ({k: st[k + "_ms"] / st["reclassifies"] for k in ("classify", "allocate", "move")}
                                    if st["reclassifies"] else None),
        "reclassifies_in_timed_region": st["reclassifies"],
        "movers_per_reclassify": st["movers"] / max(st["reclassifies"], 1),
        "move_bytes_per_reclassify": {"h2d": st["h2d_move_bytes"] / max(st["reclassifies"], 1),
                                      "d2h": st["d2h_move_bytes"] / max(st["reclassifies"], 1)},
        "tier_counts": st["tier_counts"],
        "e2e": {"value": ws * K / e2e_s, "unit": "steps/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "gpu_launches_before_timed": launches_before,
        "clocks": clocks,
        "prefill_s": prefill_s,
    }
    if rank == 0 and not args.no_cpu_baseline:
        # the oracle on one host core and on every host core (single-threaded processes)
        one = cpu_baseline(w, args.cpu_seconds, workers=1)
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds, workers=os.cpu_count() or 1)
        line["cpu_baseline"]["one_core"] = {k: one[k] for k in ("value", "cores", "sample")}
    cache.close()
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ CPU oracle
_ORACLE_CHILD = r"""
import json, sys, time
sys.path.insert(0, {root!r})
import numpy as np
from synth import WORKLOADS
from oracle import OracleCache
w = WORKLOADS[{name!r}]
budget = {budget}
# one request at the workload's full shape: prefill, then decode steps of the
# oracle as it stands, until the time budget is used
lens = w.context_lens()
order = sorted(range(w.batch), key=lambda b: lens[b])
b = order[len(order) // 2]
one = w.replace(batch=1, context=("fixed", lens[b]), n_steps=64)
oc = OracleCache.from_workload(one)
n = lens[b]
oc.append(0, one.kv_layers("k", 0, 0, n).float().numpy(), one.kv_layers("v", 0, 0, n).float().numpy(), False)
inputs = [(one.queries(t).float().numpy(), one.kv_new("k", t).float().numpy(), one.kv_new("v", t).float().numpy())
          for t in range(1, 9)]
sys.stdout.write("ready\n"); sys.stdout.flush()
sys.stdin.readline()             # all workers start timing together
t0 = time.perf_counter()
steps = 0
while time.perf_counter() - t0 < budget and steps < 64:
    steps += 1
    oc.decode_step(*inputs[(steps - 1) % len(inputs)])
el = time.perf_counter() - t0
print(json.dumps({{"seconds": el, "request_steps": steps, "tokens": n}}))
"""


def _oracle_workers(w, seconds, workers):
    """Run `workers` single-threaded oracle processes at once, each on the
    median-length request; returns their results once all are done."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    code = _ORACLE_CHILD.format(root=ROOT, name=w.name, budget=seconds)
    procs = [subprocess.Popen([sys.executable, "-c", code], stdin=subprocess.PIPE, stdout=subprocess.PIPE,
                              stderr=subprocess.PIPE, text=True, env=env) for _ in range(workers)]
    try:
        for p in procs:                       # wait until every worker has its inputs
            if p.stdout.readline().strip() != "ready":
                raise RuntimeError(p.stderr.read()[-500:])
        for p in procs:
            p.stdin.write("go\n")
            p.stdin.flush()
        out = []
        for p in procs:
            o, e = p.communicate(timeout=seconds * 10 + 600)
            if p.returncode != 0:
                raise RuntimeError(e.strip().splitlines()[-1] if e.strip() else "failed")
            out.append(json.loads(o.strip().splitlines()[-1]))
        return out
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()


def cpu_baseline(w, seconds, workers=1):
    """The oracle timed on the host: `workers` single-threaded processes at
    once, each decoding the median-length request; the batch step rate is the
    aggregate request-step rate divided by the batch size."""
    try:
        res = _oracle_workers(w, seconds, workers)
    except Exception as e:   # noqa: BLE001 - reported in the line, not raised
        return {"value": None, "unit": "steps/s", "cores": workers, "kind": "oracle", "sample": f"failed: {e}"}
    req_steps = sum(r["request_steps"] for r in res)
    wall = max(r["seconds"] for r in res)
    rate = req_steps / wall                   # request-steps per second over all workers
    return {"value": rate / w.batch, "unit": "steps/s", "cores": workers, "kind": "oracle",
            "request_steps": req_steps, "seconds": wall, "request_steps_per_s": rate,
            "batch_timed": 1, "extrapolated_to_batch": w.batch,
            "sample": f"{workers} single-threaded oracle process(es) at once, {req_steps} decode steps in all of "
                      f"one median-length request ({res[0]['tokens']} tokens, all {w.n_layers} layers) "
                      f"in {wall:.1f} s; batch step rate = request-step rate / {w.batch}"}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    w = _workload(args.workload)
    cores = os.cpu_count() or 1
    cb = cpu_baseline(w, args.cpu_seconds, workers=cores)
    v = cb["value"]
    # what was timed: request-steps (one request, all layers) on every host core
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "steps/s", "n_gpus": ws,
            "steps": cb.get("request_steps"), "step_unit": "one decode step of one request (all layers)",
            "warmup": args.warmup,
            # wall time per request-step over all cores: steps x ms_per_step = the timed seconds
            "ms_per_step": 1000.0 * cb["seconds"] / cb["request_steps"] if v else None,
            "batch_timed": 1, "extrapolated_to_batch": w.batch,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": _config(w, ws), "cpu_baseline": cb,
            "e2e": {"value": v, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _spawn_replicas(n):
    """--gpus N outside torchrun: run N replica ranks (one per GPU) under
    torch.distributed.run; rank 0 prints the line."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(29500 + os.getpid() % 1000)] + sys.argv
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--workload", default="batch32")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (profiling a small case)")
    ap.add_argument("--split-pages", type=int, default=0, help="pages per attention CTA (0: planned)")
    ap.add_argument("--host-tiers", choices=["stream", "mirror", "zerocopy"], default="stream",
                    help="T1/T2 reach attention by per-step copies (stream), a device mirror updated at "
                         "reassignment (mirror), or in place from pinned host memory (zerocopy)")
    ap.add_argument("--layers-per-launch", type=int, default=0, help="layers per attention launch (0: auto)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    ws = int(os.environ.get("WORLD_SIZE", "0"))
    if args.gpus < 1:
        sys.exit("--gpus must be >= 1")
    if ws == 0 and args.gpus > 1:
        sys.exit(_spawn_replicas(args.gpus))
    if ws and ws != args.gpus:
        sys.exit(f"--gpus {args.gpus} but WORLD_SIZE={ws}: launch one rank per GPU")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
