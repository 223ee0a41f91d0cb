"""zero3_unit_step (the unit's gather and one rank's step in one launch) against the
oracle: the gathered unit must equal the oracle's gather of the same shard bytes, and
the step's state and bf16 parameters the oracle's step, bit for bit, over two steps.
Small and ragged units run whole; the unit sweep's sizes run at full size and are
compared on the sampled windows.  Layouts that cannot take the single launch
(misaligned buffers, a shard that is not a multiple of 8) take the two-launch path,
with the same results.  Guard bands around every output check that nothing outside
the outputs is written."""
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
C16, C32 = 0x7BAD, 0x7FBADBAD
E_TIMEOUT = {v: k for k, v in za.ERRORS.items()}["ZERO_E_TIMEOUT"]


def _guarded(n, dtype, off=0):
    if dtype == torch.float32:
        base = torch.full((n + 2 * GUARD + off,), C32, dtype=torch.int32, device="cuda")
        return base, base.view(torch.float32)[GUARD + off:GUARD + off + n]
    base = torch.full((n + 2 * GUARD + off,), C16, dtype=torch.int16, device="cuda")
    return base, base[GUARD + off:GUARD + off + n]


def _intact(base, n, off=0):
    c = C32 if base.dtype == torch.int32 else C16
    return bool((base[:GUARD + off] == c).all()) and bool((base[GUARD + off + n:] == c).all())


class UnitProblem:
    """One unit (U elements, N ranks): the shards to gather and rank r's step, on the
    device and in the oracle's host mirror."""

    def __init__(self, U, N, rank=0, grad_layout=za.ZERO_GRAD_SHARD,
                 param_layout=za.ZERO_PARAM_SHARD, off=0, seed=0):
        self.U, self.N, self.rank, self.off = U, N, rank, off
        self.gl, self.pl = grad_layout, param_layout
        self.plan = plan = za.zero_plan(U, N)
        S, P = plan.shard, plan.padded
        self.S = S
        self.wl = C.StepWorkload(f"unit_step_{U}_{N}", numel=U, world=N, rank=rank, seed=seed)
        if rank < 0:
            self.lo, self.hi = 0, U
        else:
            self.lo, self.hi = rank * S, min((rank + 1) * S, U)
        self.cnt = max(0, self.hi - self.lo)
        self.sbase, self.shards = zip(*[_guarded(S, torch.int16, off) for _ in range(N)])
        for r in range(N):
            gu.dev_fill_into(self.shards[r], C.unit_shard_spec(U, N, r), 0, synth.OUT_BF16)
        self.fbase, self.full = _guarded(U, torch.int16, off)
        g_len = S if grad_layout == za.ZERO_GRAD_SHARD else P
        s_len = S if rank >= 0 else P
        p_len = S if param_layout == za.ZERO_PARAM_SHARD else U
        self.g_len, self.s_len, self.p_len = g_len, s_len, p_len
        self.gbase, self.g = zip(*[_guarded(g_len, torch.int16, off) for _ in range(N)])
        self.wbase, self.w = _guarded(s_len, torch.float32, off)
        self.mbase, self.m = _guarded(s_len, torch.float32, off)
        self.vbase, self.v = _guarded(s_len, torch.float32, off)
        self.pbase, self.p = _guarded(p_len, torch.int16, off)
        for x in (self.w, self.m, self.v):
            x.zero_()
        self.p.fill_(0x1234)
        s0 = 0 if rank < 0 else self.lo
        gu.dev_fill_into(self.w[:self.cnt if rank >= 0 else U], self.wl.master_spec(), s0,
                         synth.OUT_F32)
        self.hw = np.zeros(s_len, np.float32)
        self.hw[:self.cnt if rank >= 0 else U] = synth.fill_host(
            self.wl.master_spec(), s0, self.cnt if rank >= 0 else U, synth.OUT_F32)
        self.hm = np.zeros(s_len, np.float32)
        self.hv = np.zeros(s_len, np.float32)
        self.hp = np.full(p_len, 0x1234, np.uint16)

    def step(self, t):
        N, U, S = self.N, self.U, self.S
        host_g = []
        for k in range(N):
            self.g[k].zero_()
            spec = self.wl.grad_spec(k, t)
            if self.gl == za.ZERO_GRAD_SHARD:
                gu.dev_fill_into(self.g[k][:self.cnt], spec, self.lo, synth.OUT_BF16)
            else:
                gu.dev_fill_into(self.g[k][:U], spec, 0, synth.OUT_BF16)
            h = np.zeros(self.plan.padded, np.uint16)
            h[:U] = synth.fill_host(spec, 0, U, synth.OUT_BF16)
            host_g.append(h)
        za.zero3_unit_step(self.plan, self.rank, list(self.shards), self.full, list(self.g),
                           self.w, self.m, self.v, self.p, lr=self.wl.lr, t=t,
                           grad_layout=self.gl, param_layout=self.pl)
        # the oracle's step writes parameters by global index: give it a full buffer
        hp_full = np.zeros(U, np.uint16)
        if self.pl == za.ZERO_PARAM_FULL:
            hp_full[:] = self.hp
        else:
            hp_full[self.lo:self.hi] = self.hp[:self.cnt]
        oracle.zero_step(U, N, self.rank, host_g, self.hw, self.hm, self.hv, hp_full,
                         self.wl.lr, self.wl.beta1, self.wl.beta2, self.wl.eps, t,
                         state_base=0 if self.rank < 0 else self.lo)
        if self.pl == za.ZERO_PARAM_FULL:
            self.hp[:] = hp_full
        else:
            self.hp[:self.cnt] = hp_full[self.lo:self.hi]

    def check(self, what):
        torch.cuda.synchronize()
        host_sh = [gu.to_host_u16(x) for x in self.shards]
        for r in range(self.N):
            gu.spot_check_generated(host_sh[r], C.unit_shard_spec(self.U, self.N, r), 0,
                                    synth.OUT_BF16, samples=64, seed=r)
        assert (gu.to_host_u16(self.full) == oracle.unit_gather(self.U, self.N, host_sh)).all(), \
            f"{what}: gathered unit"
        n = self.cnt if self.rank >= 0 else self.U
        for name, d, h in (("master", self.w, self.hw), ("m", self.m, self.hm),
                           ("v", self.v, self.hv)):
            gu.assert_f32_close(gu.to_host_f32(d)[:n], h[:n], f"{what} {name}")
            assert (gu.to_host_f32(d)[n:] == 0).all(), f"{what} {name}: beyond the range"
        gu.assert_bf16_close(gu.to_host_u16(self.p), self.hp, f"{what} param")
        for b, n_ in [(x, self.S) for x in self.sbase] + [(self.fbase, self.U)] + \
                [(x, self.g_len) for x in self.gbase] + \
                [(x, self.s_len) for x in (self.wbase, self.mbase, self.vbase)] + \
                [(self.pbase, self.p_len)]:
            assert _intact(b, n_, self.off), f"{what}: a guard band was written"


# shard % 8 == 0 and aligned buffers: the single launch (register-staged step part at
# N <= 4, rank groups of 8 at 5 <= N < 40, of 32 at N >= 40); the rest: two launches
@pytest.mark.parametrize("U,N,rank", [
    (8 * 1000, 1, 0), (4096, 2, 1), (100_000, 2, 0), (96_000, 3, 2), (1 << 20, 4, 3),
    (40_000, 5, 4), (3072 * 8 * 3 + 64, 8, 0), (1_000_000, 8, 5), (2048 * 16 * 5, 16, 15),
    (33 * 8 * 1000, 33, 32), (1 << 20, 64, 0), (1 << 20, 64, 63), (100 * 8 * 333, 100, 7),
    (1_048_573, 8, 7),                      # ragged: the unit's last 5 elements, rank 7 short
    (8001, 8, 0), (100_003, 4, 1), (65_537, 8, 3),   # shard not a multiple of 8: two launches
])
def test_unit_step_matches_the_oracle(U, N, rank):
    pr = UnitProblem(U, N, rank=rank, seed=U % 97)
    for t in (1, 2):
        pr.step(t)
        pr.check(f"U={U} N={N} rank={rank} t={t}")
    assert za.device_status() == za.ZERO_OK


@pytest.mark.parametrize("layouts", [(za.ZERO_GRAD_FULL, za.ZERO_PARAM_FULL),
                                     (za.ZERO_GRAD_SHARD, za.ZERO_PARAM_FULL),
                                     (za.ZERO_GRAD_FULL, za.ZERO_PARAM_SHARD)])
@pytest.mark.parametrize("N", [4, 8, 64])
def test_unit_step_layouts(layouts, N):
    pr = UnitProblem(N * 8 * 512, N, rank=N // 2, grad_layout=layouts[0],
                     param_layout=layouts[1])
    for t in (1, 2):
        pr.step(t)
        pr.check(f"N={N} layouts {layouts} t={t}")


@pytest.mark.parametrize("N", [2, 8, 16])
def test_unit_step_all_ranks(N):
    pr = UnitProblem(N * 8 * 777, N, rank=-1, grad_layout=za.ZERO_GRAD_FULL,
                     param_layout=za.ZERO_PARAM_FULL)
    for t in (1, 2):
        pr.step(t)
        pr.check(f"N={N} all ranks t={t}")


@pytest.mark.parametrize("off", [1, 8])
@pytest.mark.parametrize("N", [2, 8])
def test_unit_step_offset_buffers(off, N):
    """Buffers 1 element off the 16-byte grid take the two launches; 8 elements off
    keep 16-byte alignment and the single launch."""
    pr = UnitProblem(N * 8 * 900, N, rank=1, off=off)
    for t in (1, 2):
        pr.step(t)
        pr.check(f"N={N} off={off} t={t}")


@pytest.mark.parametrize("U", C.UNIT_SIZES)
@pytest.mark.parametrize("N", C.UNIT_WORLDS)
def test_unit_sweep_unit_step(U, N):
    """The sweep's units at full size through zero3_unit_step, rank 0, two steps (the
    2^20 and 2^24 units as the single launch, the larger ones as two launches): the
    whole unit against the oracle's gather, the step on the sampled windows."""
    plan = za.zero_plan(U, N)
    S = plan.shard
    shards = [torch.empty(S, dtype=torch.int16, device="cuda") for _ in range(N)]
    for r in range(N):
        gu.dev_fill_into(shards[r], C.unit_shard_spec(U, N, r), 0, synth.OUT_BF16)
    full = torch.empty(U, dtype=torch.int16, device="cuda")
    wl = C.unit_workload(U, N)
    g = [torch.empty(S, dtype=torch.int16, device="cuda") for _ in range(N)]
    w = torch.empty(S, dtype=torch.float32, device="cuda")
    gu.dev_fill_into(w, wl.master_spec(), 0, synth.OUT_F32)
    m, v = torch.zeros_like(w), torch.zeros_like(w)
    p = torch.full((S,), 0x1234, dtype=torch.int16, device="cuda")
    wins = gu.sample_windows(0, S, [(0, min(S, U))], np.random.default_rng(U * 3 + N))
    wo = gu.WindowOracle(U, N, 0, wins, wl.master_spec(), (wl.lr, wl.beta1, wl.beta2, wl.eps))
    for t in (1, 2):
        full.fill_(0x5555)
        for k in range(N):
            gu.dev_fill_into(g[k], wl.grad_spec(k, t), 0, synth.OUT_BF16)
        za.zero3_unit_step(plan, 0, shards, full, g, w, m, v, p, lr=wl.lr, beta1=wl.beta1,
                           beta2=wl.beta2, eps=wl.eps, t=t)
        wo.step(t, gu.device_grad_windows(g, wins, 0, [wl.grad_spec(k, t) for k in range(N)],
                                          check_every=16, seed=t))
        torch.cuda.synchronize()
        wo.compare(w, m, v, p, 0, 0, f"unit step {U}/{N} t={t}")
    host_sh = [gu.to_host_u16(x) for x in shards]
    assert (gu.to_host_u16(full) == oracle.unit_gather(U, N, host_sh)).all()
    assert za.device_status() == za.ZERO_OK
    del shards, full, g, w, m, v, p
    torch.cuda.empty_cache()


@pytest.mark.parametrize("N", [2, 8, 64])
def test_unit_step_withheld_copies_time_out(N):
    """With the copies withheld, the single launch's waits run out: the unit is not
    written and the status word reports the timeout.  At N >= 5 the staged step part
    writes nothing either; at N <= 4 the step part reads its gradients without staging
    and completes, equal to a normal step."""
    U = N * 8 * 4096
    pr = UnitProblem(U, N, rank=0)
    ref = UnitProblem(U, N, rank=0)
    torch.cuda.synchronize()
    assert za.device_status() == za.ZERO_OK
    for k in range(N):
        gu.dev_fill_into(pr.g[k][:pr.cnt], pr.wl.grad_spec(k, 1), 0, synth.OUT_BF16)
        ref.g[k].copy_(pr.g[k])
    pr.full.fill_(-7)
    w0 = pr.w.clone()
    prev = za.test_withhold_copies(True)
    try:
        za.zero3_unit_step(pr.plan, 0, list(pr.shards), pr.full, list(pr.g), pr.w, pr.m,
                           pr.v, pr.p, lr=1e-3, t=1)
        torch.cuda.synchronize()
    finally:
        za.test_withhold_copies(prev)
    assert za.device_status() == E_TIMEOUT
    assert bool((pr.full == -7).all()), "a withheld gather wrote the unit"
    za.zero_adam_step(ref.plan, 0, list(ref.g), ref.w, ref.m, ref.v, ref.p, lr=1e-3, t=1,
                      grad_layout=za.ZERO_GRAD_SHARD, param_layout=za.ZERO_PARAM_SHARD)
    torch.cuda.synchronize()
    if N <= 4:
        assert torch.equal(pr.w, ref.w) and torch.equal(pr.p, ref.p)
    else:
        assert torch.equal(pr.w.view(torch.int32), w0.view(torch.int32))
        assert bool((pr.p == 0x1234).all())
    # the same context runs the next call normally
    za.zero3_unit_step(pr.plan, 0, list(pr.shards), pr.full, list(pr.g), pr.w, pr.m, pr.v,
                       pr.p, lr=1e-3, t=1)
    torch.cuda.synchronize()
    assert torch.equal(pr.full, torch.cat(pr.shards)[:U])
    assert za.device_status() == za.ZERO_OK


@pytest.mark.parametrize("N", [2, 8, 64])
def test_unit_step_with_host_resident_buffers(N):
    """The e2e layout: the shards, the gradient slices and the bf16 shard output in pinned
    host memory (read and written by the kernel over NVLink-C2C; the single launch's bulk
    copies read the host buffers directly).  The unit and the state must equal the
    all-device call bit for bit."""
    U = N * 8 * 4000
    dev_pr = UnitProblem(U, N, rank=1)
    host_pr = UnitProblem(U, N, rank=1)
    for k in range(N):
        gu.dev_fill_into(dev_pr.g[k][:dev_pr.cnt], dev_pr.wl.grad_spec(k, 1), dev_pr.lo,
                         synth.OUT_BF16)
    hs = [torch.empty(dev_pr.S, dtype=torch.int16, pin_memory=True) for _ in range(N)]
    hg = [torch.empty(dev_pr.S, dtype=torch.int16, pin_memory=True) for _ in range(N)]
    hp = torch.full((dev_pr.S,), 0x1234, dtype=torch.int16, pin_memory=True)
    for k in range(N):
        hs[k].copy_(dev_pr.shards[k])
        hg[k].copy_(dev_pr.g[k])
    torch.cuda.synchronize()
    za.zero3_unit_step(dev_pr.plan, 1, list(dev_pr.shards), dev_pr.full, list(dev_pr.g),
                       dev_pr.w, dev_pr.m, dev_pr.v, dev_pr.p, lr=1e-3, t=1)
    za.zero3_unit_step(host_pr.plan, 1, hs, host_pr.full, hg, host_pr.w, host_pr.m, host_pr.v,
                       hp, lr=1e-3, t=1)
    torch.cuda.synchronize()
    assert torch.equal(dev_pr.full, host_pr.full)
    for a, b in ((dev_pr.w, host_pr.w), (dev_pr.m, host_pr.m), (dev_pr.v, host_pr.v)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.equal(dev_pr.p.cpu(), hp)
    assert za.device_status() == za.ZERO_OK


@pytest.mark.parametrize("N", [2, 8, 64])
def test_unit_steps_captured_in_a_cuda_graph(N):
    """Two units' single-launch steps captured into a CUDA graph after their first eager
    call, replayed, and compared with the same calls made eagerly."""
    U = N * 8 * 3000
    a, b = UnitProblem(U, N, rank=0, seed=1), UnitProblem(U, N, rank=N - 1, seed=2)
    for pr in (a, b):
        for k in range(N):
            gu.dev_fill_into(pr.g[k][:pr.cnt], pr.wl.grad_spec(k, 1), pr.lo, synth.OUT_BF16)
    ea, eb = UnitProblem(U, N, rank=0, seed=1), UnitProblem(U, N, rank=N - 1, seed=2)
    for pr, src in ((ea, a), (eb, b)):
        for k in range(N):
            pr.g[k].copy_(src.g[k])

    def run(prs, t, stream=None):
        for pr in prs:
            za.zero3_unit_step(pr.plan, pr.rank, list(pr.shards), pr.full, list(pr.g), pr.w,
                               pr.m, pr.v, pr.p, lr=1e-3, t=t, stream=stream)

    run((a, b), 1)                          # first calls (per-device set-up) outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            run((a, b), 2)
    graph.replay()
    torch.cuda.synchronize()
    for t in (1, 2):
        run((ea, eb), t)
    torch.cuda.synchronize()
    for g_, e_ in ((a, ea), (b, eb)):
        assert torch.equal(g_.full, e_.full)
        for x, y in ((g_.w, e_.w), (g_.m, e_.m), (g_.v, e_.v)):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32))
        assert torch.equal(g_.p, e_.p)
    assert za.device_status() == za.ZERO_OK
