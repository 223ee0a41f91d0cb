"""ZeRO-2 bucketed step (zero_adam_step_range) and the gradient variants, on the GPU.

Buckets that tile the flat vector must give exactly the whole step (the step is
elementwise), whether each bucket's gradients sit in the full buffers or in
bucket-sized buffers that are reused (the full gradient never exists), and
whether the buckets run on a side stream as an emulated backward pass
produces them.  The fp32-gradient and bf16-accumulation variants are compared
with the oracle's.
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

LR, B1, B2, EPS = 1e-3, 0.9, 0.999, 1e-8


def _gspec(k, t, seed=0, zero_frac=0.0):
    return synth.Spec(seed=seed, stream=C.STREAM_GRAD, rank=k, step=t, sigma=1e-3,
                      zero_frac=zero_frac)


def _mspec(seed=0):
    return synth.Spec(seed=seed, stream=C.STREAM_MASTER, sigma=0.02)


def _state(plan, numel):
    w = torch.zeros(plan.padded, dtype=torch.float32, device="cuda")
    gu.dev_fill_into(w[:numel], _mspec(), 0, synth.OUT_F32)
    return w, torch.zeros_like(w), torch.zeros_like(w), torch.zeros(numel, dtype=torch.int16,
                                                                    device="cuda")


def _same(a, b):
    return torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a,
                       b.view(torch.int32) if b.dtype == torch.float32 else b)


@pytest.mark.parametrize("numel,world,bucket", [(1_000_003, 4, 65_537), (262_147, 16, 8_192),
                                                (100_000, 3, 99_999), (5_000, 64, 17)])
def test_buckets_tile_the_whole_step(numel, world, bucket):
    plan = za.zero_plan(numel, world)
    g = [torch.zeros(plan.padded, dtype=torch.int16, device="cuda") for _ in range(world)]
    whole = _state(plan, numel)
    buck = _state(plan, numel)
    bw = [torch.empty(bucket, dtype=torch.int16, device="cuda") for _ in range(world)]
    for t in (1, 2):
        for k in range(world):
            gu.dev_fill_into(g[k][:numel], _gspec(k, t), 0, synth.OUT_BF16)
        za.zero_adam_step(plan, -1, g, *whole, lr=LR, t=t)
        # buckets in backward order (last first), each with bucket-sized gradient buffers
        starts = list(range(0, numel, bucket))[::-1]
        for b0 in starts:
            n = min(bucket, numel - b0)
            for k in range(world):
                gu.dev_fill_into(bw[k][:n], _gspec(k, t), b0, synth.OUT_BF16)
            za.zero_adam_step_range(plan, -1, b0, b0 + bucket, bw, *buck, lr=LR, t=t)
        torch.cuda.synchronize()
        for a, b in zip(whole, buck):
            assert _same(a, b), f"t={t}"
    # and the whole step is the oracle's
    hw = np.zeros(plan.padded, np.float32)
    hw[:numel] = synth.fill_host(_mspec(), 0, numel, synth.OUT_F32)
    hm, hv, hp = np.zeros_like(hw), np.zeros_like(hw), np.zeros(numel, np.uint16)
    for t in (1, 2):
        hg = [np.pad(synth.fill_host(_gspec(k, t), 0, numel, synth.OUT_BF16),
                     (0, plan.padded - numel)) for k in range(world)]
        gu.oracle_step_parallel(numel, world, -1, hg, hw, hm, hv, hp, LR, B1, B2, EPS, t)
    gu.assert_f32_close(gu.to_host_f32(buck[0])[:numel], hw[:numel], "bucketed master")
    gu.assert_bf16_close(gu.to_host_u16(buck[3]), hp, "bucketed param")


@pytest.mark.parametrize("layout", [za.ZERO_GRAD_FULL, za.ZERO_GRAD_SHARD, za.ZERO_GRAD_WINDOW])
def test_single_rank_windows(layout):
    """Rank 1 of 4 (shard starts at an odd index), windows that straddle its range."""
    numel, world, r = 1_000_003, 4, 1
    plan = za.zero_plan(numel, world)
    S = plan.shard
    lo, hi = r * S, min((r + 1) * S, numel)
    wins = [(lo - 100, lo + 1000), (lo + 1000, lo + 77_777), (lo + 77_777, hi + 5)]
    w = torch.empty(S, dtype=torch.float32, device="cuda")
    gu.dev_fill_into(w, _mspec(), lo, synth.OUT_F32)
    m, v = torch.zeros_like(w), torch.zeros_like(w)
    p = torch.full((numel,), 0x1234, dtype=torch.int16, device="cuda")
    for b0, b1 in wins:
        if layout == za.ZERO_GRAD_FULL:
            gs = [torch.zeros(plan.padded, dtype=torch.int16, device="cuda") for _ in range(world)]
            for k in range(world):
                gu.dev_fill_into(gs[k][:numel], _gspec(k, 1), 0, synth.OUT_BF16)
        elif layout == za.ZERO_GRAD_SHARD:
            gs = [torch.zeros(S, dtype=torch.int16, device="cuda") for _ in range(world)]
            for k in range(world):
                gu.dev_fill_into(gs[k][:hi - lo], _gspec(k, 1), lo, synth.OUT_BF16)
        else:
            gs = [torch.zeros(b1 - b0, dtype=torch.int16, device="cuda") for _ in range(world)]
            for k in range(world):
                a, b = max(b0, lo), min(b1, hi)   # only the rank's part is read
                gu.dev_fill_into(gs[k][a - b0:b - b0], _gspec(k, 1), a, synth.OUT_BF16)
        za.zero_adam_step_range(plan, r, b0, b1, gs, w, m, v, p, lr=LR, t=1, grad_layout=layout)
    torch.cuda.synchronize()
    hw = synth.fill_host(_mspec(), lo, S, synth.OUT_F32)
    hw[hi - lo:] = 0
    hm, hv = np.zeros(S, np.float32), np.zeros(S, np.float32)
    hp = np.full(numel, 0x1234, np.uint16)
    hg = [np.pad(synth.fill_host(_gspec(k, 1), 0, numel, synth.OUT_BF16),
                 (0, plan.padded - numel)) for k in range(world)]
    oracle.zero_step(numel, world, r, hg, hw, hm, hv, hp, LR, B1, B2, EPS, 1, state_base=lo)
    gu.assert_f32_close(gu.to_host_f32(w)[:hi - lo], hw[:hi - lo], "rank-1 windows master")
    gu.assert_f32_close(gu.to_host_f32(m)[:hi - lo], hm[:hi - lo], "rank-1 windows m")
    dp = gu.to_host_u16(p)
    gu.assert_bf16_close(dp[lo:hi], hp[lo:hi], "rank-1 windows param")
    assert (dp[:lo] == 0x1234).all() and (dp[hi:] == 0x1234).all()


@pytest.mark.parametrize("step_streams", [1, 2])
def test_bucketed_schedule_on_a_side_stream(step_streams):
    """An emulated backward pass on stream A writes bucket gradients into a pool of two
    bucket buffers (last bucket first); a side stream steps each bucket once its event fires
    and hands the buffer back -- one side stream, or two taking the buckets in turn (bucket
    i and pool slot i % 2 on side stream i % 2).  The result equals one whole step bit for
    bit."""
    numel, world, bucket = 2_000_003, 8, 1 << 18
    plan = za.zero_plan(numel, world)
    whole = _state(plan, numel)
    buck = _state(plan, numel)
    g = [torch.zeros(plan.padded, dtype=torch.int16, device="cuda") for _ in range(world)]
    for k in range(world):
        gu.dev_fill_into(g[k][:numel], _gspec(k, 1), 0, synth.OUT_BF16)
    za.zero_adam_step(plan, -1, g, *whole, lr=LR, t=1)
    torch.cuda.synchronize()

    sa = torch.cuda.Stream()
    side = [torch.cuda.Stream() for _ in range(step_streams)]
    pool = [[torch.empty(bucket, dtype=torch.int16, device="cuda") for _ in range(world)]
            for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]
    for slot, e in enumerate(free):
        e.record(side[slot % step_streams])
    starts = list(range(0, numel, bucket))[::-1]
    for i, b0 in enumerate(starts):
        slot = i % 2
        sb = side[slot % step_streams]
        n = min(bucket, numel - b0)
        ready = torch.cuda.Event()
        with torch.cuda.stream(sa):
            sa.wait_event(free[slot])
            for k in range(world):
                synth.fill_dev(_gspec(k, 1), b0, n, synth.OUT_BF16, pool[slot][k].data_ptr(),
                               sa.cuda_stream)
            ready.record(sa)
        with torch.cuda.stream(sb):
            sb.wait_event(ready)
            za.zero_adam_step_range(plan, -1, b0, b0 + n, pool[slot], *buck, lr=LR, t=1,
                                    stream=sb)
            free[slot].record(sb)
    torch.cuda.synchronize()
    for a, b in zip(whole, buck):
        assert _same(a, b)


@pytest.mark.parametrize("world", [1, 3, 4, 8, 16, 64, 65])
@pytest.mark.parametrize("grad_f32,acc_bf16", [(True, False), (False, True), (True, True)])
@pytest.mark.parametrize("zero_frac", [0.0, 0.1])
def test_gradient_variants_vs_oracle(world, grad_f32, acc_bf16, zero_frac):
    """The f4 variants against the oracle's, with and without a tenth of the gradient sums
    exactly zero (a mask shared by the ranks: the zero shortcuts of Adam's divisions and,
    at N = 3 and 65, of the average's division)."""
    numel = 70_001
    plan = za.zero_plan(numel, world)
    kind = synth.OUT_F32 if grad_f32 else synth.OUT_BF16
    dt = torch.float32 if grad_f32 else torch.int16
    g = [torch.zeros(plan.padded, dtype=dt, device="cuda") for _ in range(world)]
    w, m, v, p = _state(plan, numel)
    flags = (za.ZERO_GRAD_F32 if grad_f32 else 0) | (za.ZERO_ACC_BF16 if acc_bf16 else 0)
    hw = np.zeros(plan.padded, np.float32)
    hw[:numel] = synth.fill_host(_mspec(), 0, numel, synth.OUT_F32)
    hm, hv, hp = np.zeros_like(hw), np.zeros_like(hw), np.zeros(numel, np.uint16)
    for t in (1, 2):
        hg = []
        for k in range(world):
            gu.dev_fill_into(g[k][:numel], _gspec(k, t, zero_frac=zero_frac), 0, kind)
            h = synth.fill_host(_gspec(k, t, zero_frac=zero_frac), 0, numel, kind)
            hg.append(np.pad(h, (0, plan.padded - numel)))
        za.zero_adam_step(plan, -1, g, w, m, v, p, lr=LR, t=t, grad_layout=flags)
        oracle.zero_step(numel, world, -1, hg, hw, hm, hv, hp, LR, B1, B2, EPS, t,
                         grad_f32=grad_f32, acc_bf16=acc_bf16)
    torch.cuda.synchronize()
    what = f"N={world} f32={grad_f32} bf16acc={acc_bf16} zeros={zero_frac}"
    gu.assert_f32_close(gu.to_host_f32(w)[:numel], hw[:numel], what + " master")
    gu.assert_f32_close(gu.to_host_f32(m)[:numel], hm[:numel], what + " m")
    gu.assert_f32_close(gu.to_host_f32(v)[:numel], hv[:numel], what + " v")
    gu.assert_bf16_close(gu.to_host_u16(p), hp, what + " param")
