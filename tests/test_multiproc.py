"""The N>1 path of bench.py on CPU with two gloo ranks: each rank routes its
own seeded batch (same shapes, different data; no collective on routed
data), and the only collective, the max-over-ranks of the timed region,
returns the slowest rank's time on every rank."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys

    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, dist, torch.device("cpu"))
    r, _ = bench.rank_workload(rank)
    out.put((rank, slowest, r.top_expert[:64].tolist(), (r.T, r.H, r.E, r.K)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    res = sorted(q.get(timeout=300) for _ in range(world))
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    assert [x[1] for x in res] == [15.0, 15.0]  # every rank sees the slowest time
    assert res[0][3] == res[1][3] == (8192, 7168, 256, 8)  # same shapes
    assert res[0][2] != res[1][2]  # different routed data per rank


def test_weak_scaling_value():
    import sys

    sys.path.insert(0, ROOT)
    import bench

    assert bench.weak_scaling_value(1, 65536, 10, 1000.0) == 655360.0
    assert bench.weak_scaling_value(4, 65536, 10, 1000.0) == 4 * 655360.0
    assert bench.max_over_ranks(3.5, None, None) == 3.5
