"""The N>1 path of bench.py on CPU: two gloo ranks, each timing its own replica.

The streaming path has no exchange step, so N GPUs run N independent
replicas; the only cross-rank operations are the barriers around the timed
region and the max over ranks of the elapsed time. These run here as a
world_size-2 gloo group on CPU."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, local = bench._dist()
    dist.barrier()
    elapsed = bench.max_over_ranks(0.5 + rank, torch.device("cpu"))
    dist.barrier()
    q.put((r, w, local, elapsed, bench.aggregate_throughput(10.0, elapsed, w)))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1] and all(o[1] == 2 for o in out)
    # both ranks see the slower rank's time; throughput counts both replicas' units
    assert all(o[3] == 1.5 for o in out)
    assert all(abs(o[4] - 2 * 10.0 / 1.5) < 1e-12 for o in out)


def test_single_process_is_untouched():
    import bench
    assert bench.max_over_ranks(0.25, torch.device("cpu")) == 0.25
    assert bench.aggregate_throughput(3.0, 2.0, 1) == 1.5
