"""Multi-GPU runs are replicas only: every rank runs an independent copy of the
workload and the job's throughput is all ranks' units over the slowest rank's
time.  The host-side logic of that (seeds, max over ranks, aggregation) runs
here on CPU with two gloo ranks."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as tmp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t_ms = 10.0 + 5.0 * rank                     # rank 1 is the slow one
    t_max = bench.max_over_ranks(t_ms, dist, "cpu")
    seeds = [None] * world
    dist.all_gather_object(seeds, bench.replica_seed_offset(rank))
    rate = bench.whole_job_rate(100.0, world, t_max)
    q.put((rank, t_max, seeds, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_over_slowest_rank():
    world = 2
    ctx = tmp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t_max, seeds, rate in out:
        assert t_max == 15.0                       # max over ranks, seen by every rank
        assert len(set(seeds)) == world            # independent problems per rank
        assert abs(rate - 2 * 100.0 / 0.015) < 1e-6


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_rate(10.0, 1, 1000.0) == 10.0
