"""The N>1 benchmark path on CPU: two gloo ranks, max-over-ranks timing and the
whole-job aggregate (replicas only: no data-path collective)."""
import os
import socket

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


def test_single_rank_aggregate():
    import bench
    ms, val = bench.aggregate(4.0, 8_000_000, 1)
    assert ms == 4.0 and val == pytest.approx(2.0)
