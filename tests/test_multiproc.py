"""The multi-GPU path of the bench on CPU: two gloo ranks, each with its own
replica workload, timing reduced with a max over ranks and whole-job
throughput computed from it (the per-token path has no exchange step, so
nothing else crosses ranks)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from synth import WORKLOADS
    w = bench.rank_workload(WORKLOADS["v32_h32_16k"], rank)
    ms = 10.0 + 5.0 * rank                 # rank 1 is the slow one
    m = bench.max_over_ranks(ms, dist)
    thr = bench.job_throughput(w.T, world, m)
    dist.barrier()
    q.put((rank, w.seed, m, thr))
    dist.destroy_process_group()


def test_two_rank_replicas_max_timing():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, m0, t0), (r1, s1, m1, t1) = res
    assert s0 != s1                         # each rank its own chunk
    assert m0 == m1 == 15.0                 # max over ranks
    assert t0 == t1 == pytest.approx(2 * 16384 / 0.015)


def test_single_process_helpers():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(100, 1, 1000.0) == 100.0
