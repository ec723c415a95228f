"""Replica timing across ranks, on CPU with the gloo backend (world size 2).

The decode step partitions by request: each rank serves its own requests and
no step exchanges data. The only cross-rank work is the bench's timing: a
barrier around the timed region, the maximum of the ranks' times, and the
whole-job throughput N * K / max time. These tests run that code path in two
gloo processes.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out_path):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    ws, r, local = bench._dist()
    assert (ws, r, local) == (world, rank, rank)
    bench._barrier(ws)
    ms = bench._max_over_ranks(ws, times[rank], torch.device("cpu"))
    bench._barrier(ws)
    dist.destroy_process_group()
    with open(f"{out_path}.{rank}", "w") as f:
        f.write(repr(ms))


def test_max_over_two_gloo_ranks(tmp_path):
    world, port = 2, _free_port()
    times = [12.5, 31.25]
    out = str(tmp_path / "ms")
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = [float(open(f"{out}.{r}").read()) for r in range(world)]
    assert got == [max(times)] * world


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench._max_over_ranks(1, 7.0, None) == 7.0
    bench._barrier(1)


if __name__ == "__main__":
    pytest.main([__file__, "-q"])


def test_bench_refuses_a_gpu_count_that_does_not_match_the_ranks():
    import subprocess
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2"], capture_output=True,
                       text=True, env=env, timeout=120)
    assert r.returncode != 0 and "WORLD_SIZE=1" in r.stderr
