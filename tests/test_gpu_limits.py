"""The header's limits, reached: ZERO_MAX_WORLD = 1024 ranks (the runtime-N step kernel and
1024-entry pointer tables in the gathers' arguments) and ZERO_MAX_UNIT_TENSORS = 256 tensors
in one row-sharded unit, on the TMA copies and on the load/store kernels; every result
against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import cuda_available
import gpu_util as gu

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]

import zero_partitioned_mixed_adam_gb300 as za  # noqa: E402
from test_gpu_step import Problem  # noqa: E402

FULL, SHARD = za.ZERO_GRAD_FULL, za.ZERO_GRAD_SHARD


@pytest.mark.parametrize("numel,world", [(100_003, za.ZERO_MAX_WORLD), (50_000, 1000)])
def test_step_at_the_largest_world(numel, world):
    """1024 ranks (a power of two: g * (1/N)) and 1000 (g / N), both on the runtime-N kernel."""
    pr = Problem(numel, world, seed=world)
    for t in (1, 2):
        pr.step(t)
        pr.check(f"N={world} t={t}")
    assert za.device_status() == za.ZERO_OK


def test_step_last_rank_of_1024():
    pr = Problem(300_007, za.ZERO_MAX_WORLD, rank=za.ZERO_MAX_WORLD - 1, grad_layout=SHARD, seed=3)
    pr.step(1)
    pr.check("rank 1023")


def _flat_gather_case(U, N):
    plan = za.zero_plan(U, N)
    host = [synth.fill_host(synth.Spec(seed=N, stream=9, rank=r, sigma=0.02), 0, plan.shard,
                            synth.OUT_BF16) for r in range(N)]
    shards = [torch.from_numpy(h.view(np.int16)).cuda() for h in host]
    full = torch.full((U,), -1, dtype=torch.int16, device="cuda")
    za.zero3_unit_gather(plan, shards, full)
    torch.cuda.synchronize()
    assert (gu.to_host_u16(full) == oracle.unit_gather(U, N, host)).all()


@pytest.mark.parametrize("U", [1_024_000 + 3, 1_000_000])
def test_flat_gather_1024_ranks(U):
    """shards of 1001 and 977 elements (not multiples of 8): the load/store kernel."""
    assert -(-U // 1024) % 8 != 0
    _flat_gather_case(U, za.ZERO_MAX_WORLD)


def test_flat_gather_1024_ranks_tma():
    """shard = 1000, a multiple of 8: the TMA copy with a 1024-entry pointer table, and a
    ragged last shard (U mod 8 = 3)."""
    U = 1024 * 1000 - 5
    assert -(-U // 1024) % 8 == 0
    _flat_gather_case(U, za.ZERO_MAX_WORLD)


@pytest.mark.parametrize("cols", [8, 3])
def test_row_gather_256_tensors_1024_ranks(cols):
    """256 tensors at 1024 ranks: most row blocks are short or empty.  cols = 8 takes the
    TMA copy (every block and offset a multiple of 8 elements), cols = 3 the load/store
    kernel."""
    rng = np.random.default_rng(cols)
    shapes = [(int(r), cols) for r in rng.integers(1, 3000, za.ZERO_MAX_UNIT_TENSORS)]
    world = za.ZERO_MAX_WORLD
    shard_len, total = za.rows_layout(shapes, world)
    host = [synth.fill_host(synth.Spec(seed=cols, stream=7, rank=r, sigma=0.02), 0, shard_len,
                            synth.OUT_BF16) for r in range(world)]
    shards = [torch.from_numpy(h.view(np.int16)).cuda() for h in host]
    full = torch.full((total,), -1, dtype=torch.int16, device="cuda")
    za.zero3_unit_gather_rows(shapes, world, shards, full)
    torch.cuda.synchronize()
    assert (gu.to_host_u16(full) == oracle.unit_gather_rows(shapes, world, host)).all()
    assert za.device_status() == za.ZERO_OK
