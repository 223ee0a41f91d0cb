"""ZeRO-3 unit gather and the per-unit step (through the C ABI) against the oracle.

The gather is a copy, so the bar is bit-exactness.  Every case, the unit sweep
(U up to 2^29, N in {2, 8, 64}) included, compares the whole gathered unit with
the oracle's gather of the same shard bytes.  The unit step is rank 0's step
on its shard from N gradient slices, writing its bf16 shard, compared with the
oracle on sampled windows over two steps.
"""
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

GUARD = 256
CANARY16 = 0x7BAD


def _shards_dev(U, N, off=0):
    plan = za.zero_plan(U, N)
    bases, views = [], []
    for r in range(N):
        b = torch.full((plan.shard + off + GUARD,), CANARY16, dtype=torch.int16, device="cuda")
        v = b[off:off + plan.shard]
        gu.dev_fill_into(v, C.unit_shard_spec(U, N, r), 0, synth.OUT_BF16)
        bases.append(b)
        views.append(v)
    return plan, bases, views


def _shards_host(U, N, S):
    return [synth.fill_host(C.unit_shard_spec(U, N, r), 0, S, synth.OUT_BF16) for r in range(N)]


# shard % 8 == 0 (with aligned buffers) takes the TMA copy: (4096, 2), (1 << 20, 64), and
# ragged units with a tail of U mod 8 elements, (7995, 8) and (163_837, 5), and empty
# trailing shards, (113, 16); the rest take the load/store kernel
@pytest.mark.parametrize("U,N", [(1, 1), (1, 4), (7, 3), (8, 8), (100, 9), (1001, 3), (4096, 2),
                                 (65537, 8), (100_000, 64), (123_457, 65), (1 << 20, 64),
                                 (7995, 8), (163_837, 5), (113, 16), (3 * 8192 * 152 + 8, 1)])
def test_gather_small_whole_unit(U, N):
    plan, bases, shards = _shards_dev(U, N)
    fb = torch.full((U + 2 * GUARD,), CANARY16, dtype=torch.int16, device="cuda")
    full = fb[GUARD:GUARD + U]
    za.zero3_unit_gather(plan, shards, full)
    torch.cuda.synchronize()
    ref = oracle.unit_gather(U, N, _shards_host(U, N, plan.shard))
    assert (gu.to_host_u16(full) == ref).all()
    assert bool((fb[:GUARD] == CANARY16).all()) and bool((fb[GUARD + U:] == CANARY16).all())


@pytest.mark.parametrize("off_src,off_dst", [(1, 0), (0, 1), (3, 5), (4, 4), (8, 8), (8, 0),
                                             (0, 4)])
def test_gather_misaligned(off_src, off_dst):
    """shard = 12,504 (a multiple of 8): offsets of 8 elements keep 16-byte alignment
    (TMA copy, with a 5-element tail); the others do not (load/store kernel)."""
    U, N = 50_013, 4
    plan, bases, shards = _shards_dev(U, N, off=off_src)
    fb = torch.full((U + off_dst + GUARD,), CANARY16, dtype=torch.int16, device="cuda")
    full = fb[off_dst:off_dst + U]
    za.zero3_unit_gather(plan, shards, full)
    torch.cuda.synchronize()
    ref = oracle.unit_gather(U, N, _shards_host(U, N, plan.shard))
    assert (gu.to_host_u16(full) == ref).all()
    assert bool((fb[:off_dst] == CANARY16).all()) and bool((fb[off_dst + U:] == CANARY16).all())


@pytest.mark.parametrize("U", C.UNIT_SIZES)
@pytest.mark.parametrize("N", C.UNIT_WORLDS)
def test_unit_sweep_gather_and_step(U, N):
    """The sweep's configuration: gather the N parameter shards, then rank 0's step on
    its shard from N gradient slices (ZERO_GRAD_SHARD, ZERO_PARAM_SHARD), two steps.

    The whole gathered unit is compared with the oracle's gather of the same shard
    bytes (host copies of the device generator's output, spot-checked against the host
    generator).  The step is compared with the oracle after t = 1 and t = 2 on the
    sampled windows of rank 0's shard: every element of 3 random 2^24 chunks, the first
    and last 2^20 elements, +-16 around its ends."""
    plan, bases, shards = _shards_dev(U, N)
    S = plan.shard
    full = torch.empty(U, dtype=torch.int16, device="cuda")
    za.zero3_unit_gather(plan, shards, full)
    torch.cuda.synchronize()
    host_sh = []
    for r, sh in enumerate(shards):
        h = gu.to_host_u16(sh)
        gu.spot_check_generated(h, C.unit_shard_spec(U, N, r), 0, synth.OUT_BF16, samples=256,
                                seed=r)
        host_sh.append(h)
    ref = oracle.unit_gather(U, N, host_sh)
    assert (gu.to_host_u16(full) == ref).all()
    del full, bases, shards, host_sh, ref

    # rank 0's step on its shard
    wl = C.unit_workload(U, N)
    g = [torch.empty(S, dtype=torch.int16, device="cuda") for _ in range(N)]
    w = torch.empty(S, dtype=torch.float32, device="cuda")
    gu.dev_fill_into(w, wl.master_spec(), 0, synth.OUT_F32)
    m = torch.zeros_like(w)
    v = torch.zeros_like(w)
    p = torch.full((S,), 0x1234, dtype=torch.int16, device="cuda")
    wins = gu.sample_windows(0, S, [(0, min(S, U))], np.random.default_rng(U + N))
    wo = gu.WindowOracle(U, N, 0, wins, wl.master_spec(), (wl.lr, wl.beta1, wl.beta2, wl.eps))
    for t in (1, 2):
        for k in range(N):
            gu.dev_fill_into(g[k], wl.grad_spec(k, t), 0, synth.OUT_BF16)
        za.zero_adam_step(plan, 0, g, w, m, v, p, lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2,
                          eps=wl.eps, t=t, grad_layout=za.ZERO_GRAD_SHARD,
                          param_layout=za.ZERO_PARAM_SHARD)
        wo.step(t, gu.device_grad_windows(g, wins, 0, [wl.grad_spec(k, t) for k in range(N)],
                                          check_every=16, seed=t))
        torch.cuda.synchronize()
        wo.compare(w, m, v, p, 0, 0, f"unit {U}/{N} t={t}")
    assert za.device_status() == za.ZERO_OK
    del g, w, m, v, p
    torch.cuda.empty_cache()


def _rows_problem(shapes, world, seed, off=0):
    shard_len, total = za.rows_layout(shapes, world)
    host = [synth.fill_host(synth.Spec(seed=seed, stream=7, rank=r, sigma=0.02), 0, shard_len,
                            synth.OUT_BF16) for r in range(world)]
    dev = []
    for r in range(world):
        b = torch.full((shard_len + off + GUARD,), CANARY16, dtype=torch.int16, device="cuda")
        v = b[off:off + shard_len]
        v.copy_(torch.from_numpy(host[r].view(np.int16)))
        dev.append(v)
    return host, dev, total


LLAMA_LAYER = [(4096, 4096)] * 4 + [(11008, 4096), (11008, 4096), (4096, 11008), (4096, 1),
                                     (4096, 1)]


# Layouts whose tensor offsets and per-rank row blocks are multiples of 8 elements take the
# TMA copy: [(64, 10)] x 8, the 256-column mix, and the last one (a short last run, an empty
# one for (9, 8), and a 4-element tail for (37, 4)); the others the load/store kernel.
@pytest.mark.parametrize("shapes,world", [
    ([(10, 3)], 4), ([(7, 5), (1, 9), (13, 1)], 3), ([(3, 2)], 8), ([(64, 10)], 8),
    ([(1000, 17), (999, 33), (5, 1)], 16), ([(300, 7)] * 20, 64), ([(257, 129)], 65),
    ([(4096, 256), (11008, 256), (256, 1)], 8),
    ([(1001, 8), (77, 16), (9, 8), (37, 4)], 4),
])
def test_gather_rows_vs_oracle(shapes, world):
    host, dev, total = _rows_problem(shapes, world, seed=len(shapes) * 100 + world)
    fb = torch.full((total + 2 * GUARD,), CANARY16, dtype=torch.int16, device="cuda")
    full = fb[GUARD:GUARD + total]
    za.zero3_unit_gather_rows(shapes, world, dev, full)
    torch.cuda.synchronize()
    ref = oracle.unit_gather_rows(shapes, world, host)
    assert (gu.to_host_u16(full) == ref).all()
    assert bool((fb[:GUARD] == CANARY16).all()) and bool((fb[GUARD + total:] == CANARY16).all())


@pytest.mark.parametrize("off", [1, 3])
def test_gather_rows_misaligned(off):
    shapes, world = [(1001, 7), (33, 3)], 4
    host, dev, total = _rows_problem(shapes, world, seed=5, off=off)
    full = torch.empty(total + 1, dtype=torch.int16, device="cuda")[1:]
    za.zero3_unit_gather_rows(shapes, world, dev, full)
    torch.cuda.synchronize()
    assert (gu.to_host_u16(full) == oracle.unit_gather_rows(shapes, world, host)).all()


@pytest.mark.parametrize("world", [2, 8, 64])
def test_gather_rows_llama_layer(world):
    """One Llama-7B layer (4 attention 4096x4096, 3 MLP 11008x4096 / 4096x11008, 2 norms)
    sharded by rows: the whole unit is compared with an independent device
    reconstruction (torch concatenation of the row blocks) and, for N <= 8, with the
    oracle on the host."""
    shard_len, total = za.rows_layout(LLAMA_LAYER, world)
    assert total == 202_383_360
    shards = [torch.empty(shard_len, dtype=torch.int16, device="cuda") for _ in range(world)]
    for r in range(world):
        gu.dev_fill_into(shards[r], synth.Spec(seed=world, stream=7, rank=r, sigma=0.02), 0,
                         synth.OUT_BF16)
    full = torch.empty(total, dtype=torch.int16, device="cuda")
    za.zero3_unit_gather_rows(LLAMA_LAYER, world, shards, full)
    parts, off = [], 0
    for rows, cols in LLAMA_LAYER:
        R = -(-rows // world)
        chunks = [s[off:off + R * cols].view(R, cols) for s in shards]
        parts.append(torch.cat(chunks)[:rows].reshape(-1))
        off += R * cols
    assert torch.equal(full, torch.cat(parts))
    torch.cuda.synchronize()
    if world <= 8:
        host = [gu.to_host_u16(s) for s in shards]
        assert (gu.to_host_u16(full) == oracle.unit_gather_rows(LLAMA_LAYER, world, host)).all()
    del shards, full, parts
    torch.cuda.empty_cache()
