"""Pin: the oracle against the method run as it is meant to run -- N processes and real
collectives.  Four gloo ranks on CPU each hold their fp32 shard of the master weights and of
m, v; every step they reduce-scatter their fp32 gradients (a sum), divide by N, update their
shard with bias-corrected Adam in fp32, and all-gather the shards back into the full vector
("ZeRO and FSDP" -> "Implementing ZeRO's Adam from scratch": the optimizer step of ZeroAdam,
restated here in plain torch ops).  gloo's summation order is not documented and torch's
fused `add_(alpha=)` / `addcmul_` may round differently, so the reduced gradient and the
moments can differ from the oracle's (fp32-gradient variant, rank-order sum) in their last
bits; where a value crosses zero that is an unbounded relative error.  The bar is therefore
normwise: every element within 1e-6 of its array's largest magnitude (measured: a few ulps,
3.7e-8 on weights of up to 0.10)."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle

NUMEL, WORLD, STEPS = 10_007, 4, 3
LR, B1, B2, EPS = 1e-2, 0.9, 0.999, 1e-8


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    rng = np.random.default_rng(2024)
    w0 = rng.normal(0, 0.02, NUMEL).astype(np.float32)
    grads = [[rng.normal(0, 1e-3, NUMEL).astype(np.float32) for _ in range(WORLD)]
             for _ in range(STEPS)]
    return w0, grads


def _rank(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    torch.set_num_threads(1)
    w0, grads = _inputs()
    shard = -(-NUMEL // WORLD)
    padded = shard * WORLD
    full = torch.zeros(padded, dtype=torch.float32)
    full[:NUMEL] = torch.from_numpy(w0)
    master = full[rank * shard:(rank + 1) * shard].clone()   # this rank's fp32 shard
    m = torch.zeros(shard, dtype=torch.float32)
    v = torch.zeros(shard, dtype=torch.float32)
    for t in range(1, STEPS + 1):
        flat = torch.zeros(padded, dtype=torch.float32)
        flat[:NUMEL] = torch.from_numpy(grads[t - 1][rank])
        g = torch.empty(shard, dtype=torch.float32)
        dist.reduce_scatter_tensor(g, flat)                   # sum over the ranks
        g /= WORLD
        m.mul_(B1).add_(g, alpha=1 - B1)
        v.mul_(B2).addcmul_(g, g, value=1 - B2)
        m_hat = m / (1 - B1 ** t)
        v_hat = v / (1 - B2 ** t)
        master -= LR * m_hat / (v_hat.sqrt() + EPS)
        dist.all_gather_into_tensor(full, master)
    ms = [torch.empty(shard) for _ in range(WORLD)]
    vs = [torch.empty(shard) for _ in range(WORLD)]
    dist.all_gather(ms, m)
    dist.all_gather(vs, v)
    if rank == 0:
        out["w"] = full[:NUMEL].numpy().copy()
        out["m"] = torch.cat(ms)[:NUMEL].numpy().copy()
        out["v"] = torch.cat(vs)[:NUMEL].numpy().copy()
    dist.barrier()
    dist.destroy_process_group()


def test_oracle_matches_four_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_rank, args=(_free_port(), out), nprocs=WORLD, start_method="spawn")
    w0, grads = _inputs()
    P = -(-NUMEL // WORLD) * WORLD
    hw = np.zeros(P, np.float32)
    hw[:NUMEL] = w0
    hm, hv = np.zeros(P, np.float32), np.zeros(P, np.float32)
    hp = np.zeros(NUMEL, np.uint16)
    for t in range(1, STEPS + 1):
        g = [np.pad(x, (0, P - NUMEL)) for x in grads[t - 1]]
        oracle.zero_step(NUMEL, WORLD, -1, g, hw, hm, hv, hp, LR, B1, B2, EPS, t, grad_f32=True)
    for name, ref, got in (("master", hw[:NUMEL], out["w"]), ("m", hm[:NUMEL], out["m"]),
                           ("v", hv[:NUMEL], out["v"])):
        # normwise: the largest difference within 1e-6 of the array's largest magnitude
        d = np.abs(got.astype(np.float64) - ref)
        assert d.max() <= 1e-6 * np.abs(ref).max(), (name, float(d.max()))
    # the weights moved by about lr per step (the updates are not vacuous)
    assert np.median(np.abs(out["w"] - w0)) > STEPS * LR * 0.5
