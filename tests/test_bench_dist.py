"""The N>1 benchmark path on CPU: two gloo ranks, max-over-ranks timing and the
whole-job aggregate (replicas only: no data-path collective), and a rank that leaves
before the aggregate: the survivor's collective must fail within the process group's
timeout instead of waiting for ever."""
import datetime
import os
import socket
import time

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms_local = [10.0, 12.5][rank]
    ms, val = bench.aggregate(ms_local, 1_000_000, world, dist, None)
    out[rank] = (ms, val)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregate_is_max_time_and_total_elements():
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn")
    for r in (0, 1):
        ms, val = out[r]
        assert ms == 12.5
        assert val == pytest.approx(2 * 1_000_000 / 12.5e-3 / 1e9)


def _worker_one_leaves(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=5))
    if rank == 1:
        out[1] = "left"
        os._exit(0)              # leaves between steps: nothing of it is in flight
    t0 = time.perf_counter()
    try:
        bench.aggregate(10.0, 1_000_000, world, dist, None)
        out[0] = ("no error", time.perf_counter() - t0)
    except Exception as e:   # gloo reports the lost peer or the timeout
        out[0] = ("error", time.perf_counter() - t0, type(e).__name__)


def test_a_rank_that_leaves_fails_the_survivor_cleanly():
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    mp.start_processes(_worker_one_leaves, args=(2, port, out), nprocs=2, start_method="spawn")
    assert out[1] == "left"
    assert out[0][0] == "error", out[0]
    assert out[0][1] < 60


def test_single_rank_aggregate():
    import bench
    ms, val = bench.aggregate(4.0, 8_000_000, 1)
    assert ms == 4.0 and val == pytest.approx(2.0)
