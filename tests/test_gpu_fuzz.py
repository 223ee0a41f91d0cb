"""Seeded random sweeps against the oracle: sizes, rank counts, single-rank or all-ranks mode,
gradient and parameter layouts, buffer misalignments (which decide between the TMA-staged and
the register-staged step kernels, and between the TMA and the load/store gathers), windows,
and gather layouts.  The cases are drawn once from a fixed seed, so every run checks the same
ones; each is compared with the oracle bit for bit (through the usual tolerance check)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import configs as C
from conftest import cuda_available
import gpu_util as gu

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]

import zero_partitioned_mixed_adam_gb300 as za  # noqa: E402
from test_gpu_step import Problem  # noqa: E402

FULL, SHARD = za.ZERO_GRAD_FULL, za.ZERO_GRAD_SHARD
WORLDS = [1, 2, 3, 4, 5, 7, 8, 8, 8, 9, 13, 16, 16, 16, 17, 31, 32, 64, 100]


def _step_cases(n=48, seed=20261202):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        world = int(rng.choice(WORLDS))
        numel = int(rng.integers(1, 300_000)) if i % 4 else int(rng.integers(world, 8 * world + 9))
        rank = -1 if rng.random() < 0.5 else int(rng.integers(0, world))
        gl = FULL if rank < 0 or rng.random() < 0.5 else SHARD
        pl = FULL if rank < 0 or rng.random() < 0.6 else SHARD
        # half the cases fully aligned (the staged kernels at N >= 5), half not
        offs = (0, 0, 0) if rng.random() < 0.5 else tuple(int(x) for x in rng.integers(0, 8, 3))
        # a third of the cases without zeros, a third with 10 %, a third with 50 % of the
        # gradient sums exactly zero (from the index: the draws above stay as they were)
        cases.append((numel, world, rank, gl, pl, offs, i, (0.0, 0.1, 0.5)[i % 3]))
    return cases


@pytest.mark.parametrize("numel,world,rank,gl,pl,offs,seed,zero_frac", _step_cases())
def test_step_sweep(numel, world, rank, gl, pl, offs, seed, zero_frac):
    pr = Problem(numel, world, rank=rank, grad_layout=gl, param_layout=pl, offs=offs, seed=seed,
                 zero_frac=zero_frac)
    for t in (1, 2):
        pr.step(t)
        pr.check(f"numel={numel} N={world} rank={rank} gl={gl} pl={pl} offs={offs} "
                 f"zeros={zero_frac} t={t}")
    assert za.device_status() == za.ZERO_OK


def _window_cases(n=12, seed=7):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        world = int(rng.choice([2, 4, 8, 16, 5, 64]))
        numel = int(rng.integers(10_000, 400_000))
        b0 = int(rng.integers(0, numel))
        b1 = int(rng.integers(b0, numel + 50))
        out.append((numel, world, b0, b1, i))
    return out


@pytest.mark.parametrize("numel,world,b0,b1,seed", _window_cases())
def test_window_sweep(numel, world, b0, b1, seed):
    """All ranks, one window [b0, b1) with its own gradient buffers (ZERO_GRAD_WINDOW): the
    window equals the oracle on it, everything outside is untouched."""
    plan = za.zero_plan(numel, world)
    P = plan.padded
    gspec = [synth.Spec(seed=seed, stream=C.STREAM_GRAD, rank=k, step=1, sigma=1e-3)
             for k in range(world)]
    mspec = synth.Spec(seed=seed, stream=C.STREAM_MASTER, sigma=0.02)
    n = max(0, min(b1, numel) - b0)
    gw = [torch.zeros(max(b1 - b0, 1), dtype=torch.int16, device="cuda") for _ in range(world)]
    for k in range(world):
        gu.dev_fill_into(gw[k][:n], gspec[k], b0, synth.OUT_BF16)
    w = torch.zeros(P, dtype=torch.float32, device="cuda")
    gu.dev_fill_into(w[:numel], mspec, 0, synth.OUT_F32)
    m, v = torch.zeros_like(w), torch.zeros_like(w)
    p = torch.full((numel,), 0x1234, dtype=torch.int16, device="cuda")
    za.zero_adam_step_range(plan, za.ZERO_ALL_RANKS, b0, b1, gw, w, m, v, p, lr=1e-3, t=1,
                            grad_layout=za.ZERO_GRAD_WINDOW)
    torch.cuda.synchronize()
    hw = np.zeros(P, np.float32)
    hw[:numel] = synth.fill_host(mspec, 0, numel, synth.OUT_F32)
    hw0 = hw.copy()
    hm, hv = np.zeros(P, np.float32), np.zeros(P, np.float32)
    hp = np.full(numel, 0x1234, np.uint16)
    if n:
        hg = [synth.fill_host(gspec[k], b0, n, synth.OUT_BF16) for k in range(world)]
        oracle.zero_step(numel, world, -1, hg, hw, hm, hv, hp, 1e-3, 0.9, 0.999, 1e-8, 1,
                         i0=b0, i1=b0 + n, grad_base=b0)
    gu.assert_f32_close(gu.to_host_f32(w), hw, "window master")
    gu.assert_f32_close(gu.to_host_f32(m), hm, "window m")
    gu.assert_f32_close(gu.to_host_f32(v), hv, "window v")
    gu.assert_bf16_close(gu.to_host_u16(p), hp, "window params")
    outside = np.ones(P, bool)
    outside[b0:b0 + n] = False
    assert (gu.to_host_f32(w)[outside] == hw0[outside]).all()


def _gather_cases(n=24, seed=11):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        world = int(rng.choice([1, 2, 3, 8, 8, 16, 64, 100]))
        if rng.random() < 0.5:   # shard a multiple of 8: the TMA copy when aligned
            S = 8 * int(rng.integers(1, 40_000 // world + 2))
            U = int(rng.integers(max(1, (world - 1) * S + 1), world * S + 1))
        else:
            U = int(rng.integers(1, 400_000))
        off_s = int(rng.choice([0, 0, 8, 1, 3]))
        off_f = int(rng.choice([0, 0, 8, 2]))
        out.append((U, world, off_s, off_f, i))
    return out


@pytest.mark.parametrize("U,world,off_s,off_f,seed", _gather_cases())
def test_flat_gather_sweep(U, world, off_s, off_f, seed):
    plan = za.zero_plan(U, world)
    host = [synth.fill_host(synth.Spec(seed=seed, stream=9, rank=r, sigma=0.02), 0, plan.shard,
                            synth.OUT_BF16) for r in range(world)]
    shards = []
    for h in host:
        b = torch.zeros(plan.shard + off_s, dtype=torch.int16, device="cuda")
        b[off_s:].copy_(torch.from_numpy(h.view(np.int16)))
        shards.append(b[off_s:])
    fb = torch.full((U + off_f + 64,), -7, dtype=torch.int16, device="cuda")
    full = fb[off_f:off_f + U]
    za.zero3_unit_gather(plan, shards, full)
    torch.cuda.synchronize()
    assert (gu.to_host_u16(full) == oracle.unit_gather(U, world, host)).all()
    assert bool((fb[:off_f] == -7).all()) and bool((fb[off_f + U:] == -7).all())
    assert za.device_status() == za.ZERO_OK


def _rows_cases(n=16, seed=13):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        world = int(rng.choice([1, 2, 4, 8, 16, 64, 65]))
        T = int(rng.integers(1, 12))
        aligned = rng.random() < 0.5   # cols a multiple of 8: every row block a multiple of 8
        shapes = [(int(rng.integers(1, 3000)),
                   8 * int(rng.integers(1, 40)) if aligned else int(rng.integers(1, 300)))
                  for _ in range(T)]
        out.append((shapes, world, i))
    return out


@pytest.mark.parametrize("shapes,world,seed", _rows_cases())
def test_row_gather_sweep(shapes, world, seed):
    shard_len, total = za.rows_layout(shapes, world)
    host = [synth.fill_host(synth.Spec(seed=seed, stream=7, rank=r, sigma=0.02), 0, shard_len,
                            synth.OUT_BF16) for r in range(world)]
    shards = [torch.from_numpy(h.view(np.int16)).cuda() for h in host]
    full = torch.full((total,), -7, dtype=torch.int16, device="cuda")
    za.zero3_unit_gather_rows(shapes, world, shards, full)
    torch.cuda.synchronize()
    assert (gu.to_host_u16(full) == oracle.unit_gather_rows(shapes, world, host)).all()
    assert za.device_status() == za.ZERO_OK


def _unit_step_cases(n=32, seed=17):
    """Units whose shard is a multiple of 8 half the time (the one-launch path when every
    buffer is aligned), any rank, both gradient and parameter layouts, and offsets that keep
    or break the 16-byte alignment."""
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        world = int(rng.choice(WORLDS))
        if i % 2:
            U = int(rng.integers(1, 40_000)) * 8 * world - int(rng.integers(0, 8))
        else:
            U = int(rng.integers(world, 300_000))
        U = max(U, 1)
        rank = int(rng.integers(0, world))
        gl = FULL if rng.random() < 0.3 else SHARD
        pl = za.ZERO_PARAM_FULL if rng.random() < 0.3 else za.ZERO_PARAM_SHARD
        off = int(rng.choice([0, 0, 0, 8, 1, 3]))
        cases.append((U, world, rank, gl, pl, off, i))
    return cases


@pytest.mark.parametrize("U,world,rank,gl,pl,off,seed", _unit_step_cases())
def test_unit_step_sweep(U, world, rank, gl, pl, off, seed):
    from test_gpu_unit_step import UnitProblem
    pr = UnitProblem(U, world, rank=rank, grad_layout=gl, param_layout=pl, off=off, seed=seed)
    for t in (1, 2):
        pr.step(t)
        pr.check(f"unit step fuzz {seed} t={t}")
    assert za.device_status() == za.ZERO_OK
