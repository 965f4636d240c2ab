"""The benchmark's multi-rank path on CPU: two gloo ranks (world size 2).

The layer runs as independent replicas (no exchange step on one replica), so what
spans ranks is host-side: the process group set up from the torchrun environment,
barriers, the max-over-ranks time, the sum of tokens/s over ranks, and distinct tokens
per rank. These run here with the gloo backend; no GPU is involved.
"""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    from mixture_experts_layer_gemv_gb300.synth import WORKLOADS, make_tokens
    dist, r, w = bench._dist()
    assert (r, w) == (rank, world) and dist.get_backend() == "gloo"
    bench._barrier(dist)
    mx = bench._max_over_ranks(dist, 1.5 + rank)       # per-rank "ms per step"
    sm = bench._sum_over_ranks(dist, 1000.0 * (rank + 1))  # per-rank tokens/s
    wl = WORKLOADS["tiny_t8"]
    x = make_tokens(wl.cfg, wl.T, bench.replica_seed(wl.seed, rank, 0), "cpu", name="x_step0")
    xs = [torch.zeros_like(x) for _ in range(world)]
    dist.all_gather(xs, x)
    distinct = not torch.equal(xs[0], xs[1])
    out[rank] = (mx, sm, distinct)
    bench._barrier(dist)
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_times_and_use_distinct_tokens():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        for p in procs:
            if p.is_alive():
                p.kill()
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        res = dict(out)
    for r in range(world):
        mx, sm, distinct = res[r]
        assert mx == 2.5          # the slowest rank's time
        assert sm == 3000.0       # whole-job throughput: sum over ranks
        assert distinct           # each replica runs its own tokens


def test_single_process_needs_no_process_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    sys.path.insert(0, ROOT)
    import bench
    dist, rank, world = bench._dist()
    assert dist is None and (rank, world) == (0, 1)
    assert bench._max_over_ranks(None, 4.0) == 4.0 and bench._sum_over_ranks(None, 7.0) == 7.0
