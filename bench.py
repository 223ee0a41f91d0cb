#!/usr/bin/env python3
"""Benchmark of the fused ZeRO-1/2 Adam step on GB300: Gelem/s and achieved HBM GB/s.

One step = one call of zero_adam_step over every rank's shard (or one rank's,
for the single-rank workload): the emulated reduce-scatter of the N ranks' bf16
gradients, bias-corrected Adam on the fp32 master/m/v, and the bf16 cast into
the flat parameter buffer.  Inputs are seeded and synthetic (synth/), resident
in HBM before timing.  A workload that moves at least four L2 sizes per step
(every default one) runs its timed steps back to back; a smaller one (tiny, the
small ZeRO-3 units) has the L2 flushed before every timed step, outside the
timed launches.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

With --gpus N > 1 (under torchrun) every rank runs an independent replica of
the workload on its own GPU (the N emulated ZeRO ranks live inside each GPU's
HBM; there is no cross-GPU exchange), and the value is all ranks' elements
over the slowest rank's time.  --impl reference times the CPU oracle on the
host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ZeRO Adam step Gelem/s and achieved HBM GB/s vs GB300 peak (1 GPU)"
FALLBACK_HBM_GBS = 6800.0
L2_FALLBACK_BYTES = 129 << 20   # GB300's L2, when the device does not report it


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _workload(name):
    from synth import configs as C
    if name in C.WORKLOADS:
        return C.WORKLOADS[name]
    if name.startswith("unit"):
        # unit:<U>:<N>
        _, u, n = name.split(":")
        return C.unit_workload(int(u), int(n))
    if name.startswith("shard:"):
        # shard:<U>:<N>: the unit's rank-0 step alone, without the gather before it
        _, u, n = name.split(":")
        return C.unit_shard_step_workload(int(u), int(n))
    raise SystemExit(f"unknown workload {name}")


def _bytes_per_step(wl, shard):
    """Algorithmic bytes of one step: (2N + 26) per stepped element ((4N + 26) with fp32
    gradients)."""
    n = _elements(wl, shard)
    return ((4 if wl.grad_f32 else 2) * wl.world + 26) * n


def _grad_flags(za, wl):
    return (za.ZERO_GRAD_F32 if wl.grad_f32 else 0) | (za.ZERO_ACC_BF16 if wl.acc_bf16 else 0)


def _elements(wl, shard):
    """Elements one step updates: all of them, or the stepped rank's real ones."""
    if wl.rank < 0:
        return wl.numel
    lo = wl.rank * shard
    return max(0, min(shard, wl.numel - lo))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        # return once the first sample is in (nvidia-smi attached and querying), so that
        # the steps that follow are sampled from their start
        deadline = time.perf_counter() + 10.0
        while not self.lines and time.perf_counter() < deadline and self.proc.poll() is None:
            time.sleep(0.01)
        time.sleep(0.1)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def code_hash(*paths):
    """SHA-256 of C++/CUDA sources with their // comments, trailing blanks and empty
    lines removed: it changes when the code does, not when a comment does."""
    lines = []
    for path in paths:
        with open(path, encoding="utf-8") as f:
            for line in f:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    lines.append(code)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()


def kernel_source_hash(kernel_src):
    """code_hash of a kernel file together with every header of the library's sources
    (the kernels' shared device code lives in them)."""
    csrc = os.path.dirname(kernel_src)
    headers = sorted(os.path.join(csrc, h) for h in os.listdir(csrc) if h.endswith(".h"))
    return code_hash(kernel_src, *headers)


def traffic_key(kernel, wl):
    """Key of a kernel's traffic record: kernel/N, and the gradient variant when it is not
    the method's bf16 gradients with an fp32 sum (other bytes per element)."""
    variant = "/f32" if wl.grad_f32 else "/bf16sum" if wl.acc_bf16 else ""
    return f"{kernel}/N{wl.world}{variant}"


def launch_traffic(kernel, wl, n):
    """DRAM bytes of one call of `kernel` (a launch, or "a+b" for a call that launches two)
    from the committed records, or None when a record is missing or void: per unit element
    for the gathers and the one-launch unit step, per stepped element (n) for the steps."""
    total = 0.0
    for k in kernel.split("+"):
        if k == "zero3_unit_step_kernel":
            src, units = "adam_step.cu", wl.numel
        elif k.startswith("zero_adam_step"):
            src, units = "adam_step.cu", n
        elif k.startswith("zero3_unit_gather"):
            src, units = "unit_gather.cu", wl.numel
        else:
            return None
        rec = _traffic_record(os.path.join(ROOT, "zero_partitioned_mixed_adam_gb300", "csrc", src))
        rec = (rec or {}).get(traffic_key(k, wl))
        if not rec:
            return None
        total += rec["dram_bytes_per_element"] * units
    return total


def _traffic_record(kernel_src):
    """DRAM traffic per element from the committed ncu summary, if it was taken on
    the current code of the kernel's source file and headers (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        return rec.get(kernel_source_hash(kernel_src))
    except Exception:
        return None


class Replica:
    """One replica's device buffers and the launches of one step.

    Step workloads: one zero_adam_step.  Unit workloads (ZeRO-3): the unit
    gather of the N parameter shards, then rank 0's step on its shard."""

    def __init__(self, wl, dev, unit_mode="fused"):
        import torch
        import synth
        import zero_partitioned_mixed_adam_gb300 as za
        self.za, self.wl, self.dev = za, wl, dev
        self.unit_mode = unit_mode
        self.plan = plan = za.zero_plan(wl.numel, wl.world)
        S, P = plan.shard, plan.padded
        single = wl.rank >= 0
        self.lo = wl.rank * S if single else 0
        self.n = n = _elements(wl, plan.shard)
        self.unit = wl.name.startswith("unit")
        g_len = S if wl.grad_layout == "shard" else P
        s_len = S if single else P
        p_len = S if wl.param_layout == "shard" else wl.numel
        self.g_first = 0 if wl.grad_layout == "shard" else self.lo
        self.p_first = 0 if wl.param_layout == "shard" else self.lo
        gdt = torch.float32 if wl.grad_f32 else torch.int16
        self.g = [torch.zeros(g_len, dtype=gdt, device=dev) for _ in range(wl.world)]
        self.g_ptrs = za.pointer_array(self.g)
        self.w = torch.zeros(s_len, dtype=torch.float32, device=dev)
        self.m = torch.zeros_like(self.w)
        self.v = torch.zeros_like(self.w)
        self.p = torch.zeros(p_len, dtype=torch.int16, device=dev)
        st = torch.cuda.current_stream(dev).cuda_stream
        synth.fill_dev(wl.master_spec(), self.lo, n, synth.OUT_F32, self.w.data_ptr(), st)
        self.shards, self.full = None, None
        if self.unit:
            from synth import configs as C
            self.shards = [torch.empty(S, dtype=torch.int16, device=dev) for _ in range(wl.world)]
            for r in range(wl.world):
                synth.fill_dev(C.unit_shard_spec(wl.numel, wl.world, r), 0, S, synth.OUT_BF16,
                               self.shards[r].data_ptr(), st)
            self.full = torch.empty(wl.numel, dtype=torch.int16, device=dev)
            self.shard_ptrs = za.pointer_array(self.shards)
        # (name, algorithmic bytes) of the step's timed calls, in order
        self.kernels = []
        if self.unit and self.unit_mode == "fused":
            self.kernels.append((self.unit_step_kernel_name(),
                                 4 * wl.numel + _bytes_per_step(wl, plan.shard)))
        else:
            if self.unit:
                self.kernels.append((self.gather_kernel_name(), 4 * wl.numel))
            self.kernels.append((self.step_kernel_name(), _bytes_per_step(wl, plan.shard)))

    def gather_kernel_name(self):
        """The library copies on the TMA engine when the shard is a multiple of 8
        elements and every buffer is 16-byte aligned (whole cudaMalloc buffers)."""
        tma = (self.wl.numel >= 8 and self.plan.shard % 8 == 0
               and all(x.data_ptr() % 16 == 0 for x in self.shards + [self.full]))
        return "zero3_unit_gather_tma_kernel" if tma else "zero3_unit_gather_kernel"

    def unit_step_kernel_name(self):
        """zero3_unit_step runs the gather and the step as one launch when the shard
        is a multiple of 8 elements, every buffer is 16-byte aligned at its first
        element and the unit moves at most 512 MiB; otherwise the gather kernel, then
        the step kernel."""
        aligned = all(x.data_ptr() % 16 == 0
                      for x in self.shards + [self.full] + self.g + [self.w, self.m, self.v,
                                                                     self.p])
        small = 4 * self.wl.numel + _bytes_per_step(self.wl, self.plan.shard) <= (512 << 20)
        plain = not (self.wl.grad_f32 or self.wl.acc_bf16)
        if (self.wl.numel >= 8 and self.n >= 8 and self.plan.shard % 8 == 0 and aligned and small
                and plain):
            return "zero3_unit_step_kernel"
        return f"{self.gather_kernel_name()}+{self.step_kernel_name()}"

    def step_kernel_name(self):
        """The library runs the TMA-staged kernel (gradients staged in rank groups)
        for N >= 5 when every buffer is 16-byte aligned at the range's first
        element (whole cudaMalloc buffers); the register-staged kernel otherwise
        (its fixed-N instance, or its any-N kernel)."""
        def aligned(t, first, esize):
            return (t.data_ptr() + first * esize) % 16 == 0
        gsize = 4 if self.wl.grad_f32 else 2
        tma = (self.wl.world >= 5 and self.n >= 8 and not self.wl.grad_f32 and not self.wl.acc_bf16
               and all(aligned(g, self.g_first, gsize) for g in self.g)
               and all(aligned(x, 0, 4) for x in (self.w, self.m, self.v))
               and aligned(self.p, self.p_first, 2))
        if tma:
            return "zero_adam_step_tma_grad_kernel"
        # the register-staged kernel: an instance per N in 1, 2, 4, ..., 64, else any-N
        return ("zero_adam_step_kernel" if self.wl.world in (1, 2, 4, 8, 16, 32, 64)
                else "zero_adam_step_any_kernel")

    def fill_grads(self, t):
        import torch
        import synth
        st = torch.cuda.current_stream(self.dev).cuda_stream
        kind, gsize = (synth.OUT_F32, 4) if self.wl.grad_f32 else (synth.OUT_BF16, 2)
        for k in range(self.wl.world):
            synth.fill_dev(self.wl.grad_spec(k, t), self.lo, self.n, kind,
                           self.g[k].data_ptr() + gsize * self.g_first, st)

    def step(self, t, stream, ev=None, grads=None, shards=None, param=None):
        """Issue one step; ev[i] = (start, end) events around launch i when given.
        grads/shards/param override the device buffers (host-resident inputs)."""
        za, wl = self.za, self.wl
        i = 0
        if self.unit and self.unit_mode == "fused":
            if ev is not None:
                ev[0][0].record(stream)
            za.zero3_unit_step(self.plan, wl.rank,
                               shards if shards is not None else self.shard_ptrs, self.full,
                               grads if grads is not None else self.g_ptrs,
                               self.w, self.m, self.v,
                               param if param is not None else self.p, lr=wl.lr,
                               beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps, t=t,
                               grad_layout=za.ZERO_GRAD_SHARD | _grad_flags(za, wl),
                               param_layout=za.ZERO_PARAM_SHARD,
                               stream=stream)
            if ev is not None:
                ev[0][1].record(stream)
            return
        if self.unit:
            if ev is not None:
                ev[i][0].record(stream)
            za.zero3_unit_gather(self.plan, shards if shards is not None else self.shard_ptrs,
                                 self.full, stream=stream)
            if ev is not None:
                ev[i][1].record(stream)
            i += 1
        if ev is not None:
            ev[i][0].record(stream)
        za.zero_adam_step(self.plan, wl.rank, grads if grads is not None else self.g_ptrs,
                          self.w, self.m, self.v,
                          param if param is not None else self.p, lr=wl.lr, beta1=wl.beta1,
                          beta2=wl.beta2, eps=wl.eps, t=t,
                          grad_layout=(za.ZERO_GRAD_SHARD if wl.grad_layout == "shard" else 0)
                          | _grad_flags(za, wl),
                          param_layout=za.ZERO_PARAM_SHARD if wl.param_layout == "shard" else 0,
                          stream=stream)
        if ev is not None:
            ev[i][1].record(stream)

    def unit_elements(self):
        """Elements one step processes: the unit's U for ZeRO-3 units, else the
        stepped parameters."""
        return self.wl.numel if self.unit else self.n

    def step_bytes(self):
        return sum(b for _, b in self.kernels)


class L2Flush:
    """Evicts the L2 between timed steps of a workload that moves less than a few L2
    sizes per step: a write of twice the L2, then a read of another such buffer, so
    that the next step starts with clean lines (no write-backs charged to it)."""

    def __init__(self, dev):
        import torch
        props = torch.cuda.get_device_properties(dev)
        l2 = getattr(props, "L2_cache_size", 0) or L2_FALLBACK_BYTES
        self.nbytes = 2 * l2
        self.a = torch.empty(self.nbytes // 4, dtype=torch.float32, device=dev)
        self.b = torch.zeros(self.nbytes // 4, dtype=torch.float32, device=dev)
        self.l2 = l2

    def __call__(self, i):
        self.a.fill_(float(i & 7))
        self.b.sum()

    @staticmethod
    def needed(step_bytes, dev):
        import torch
        props = torch.cuda.get_device_properties(dev)
        l2 = getattr(props, "L2_cache_size", 0) or L2_FALLBACK_BYTES
        return step_bytes < 4 * l2


class OracleSample:
    """The oracle (plain C) on a window of the workload, run over all host cores as
    disjoint sub-windows.  Inputs are generated once; each call steps the window."""

    def __init__(self, wl, max_elems=1 << 22):
        import numpy as np
        import synth
        self.wl = wl
        S = -(-wl.numel // wl.world)
        lo = wl.rank * S if wl.rank >= 0 else 0
        n = min(max_elems, wl.numel - lo, S if wl.rank >= 0 else wl.numel)
        self.a, self.b, self.n = lo, lo + n, n
        kind = synth.OUT_F32 if wl.grad_f32 else synth.OUT_BF16
        self.grads = [synth.fill_host(wl.grad_spec(k, wl.prewarm + 1), lo, n, kind)
                      for k in range(wl.world)]
        self.hw = synth.fill_host(wl.master_spec(), lo, n, synth.OUT_F32)
        self.hm = np.zeros(n, np.float32)
        self.hv = np.zeros(n, np.float32)
        self.hp = np.zeros(n, np.uint16)
        self.cores = os.cpu_count() or 1
        chunk = -(-n // self.cores)
        self.bounds = [(lo + i, min(lo + n, lo + i + chunk)) for i in range(0, n, chunk)]
        self.t = wl.prewarm

    def step(self):
        import oracle
        from concurrent.futures import ThreadPoolExecutor
        wl, a = self.wl, self.a
        self.t += 1
        t = self.t

        def run(ab):
            oracle.zero_step(wl.numel, wl.world, -1 if wl.rank < 0 else wl.rank, self.grads,
                             self.hw, self.hm, self.hv, self.hp, wl.lr, wl.beta1, wl.beta2,
                             wl.eps, t, i0=ab[0], i1=ab[1], grad_base=a, state_base=a,
                             param_base=a, grad_f32=wl.grad_f32,
                             acc_bf16=wl.acc_bf16)
        with ThreadPoolExecutor(max_workers=self.cores) as ex:
            list(ex.map(run, self.bounds))

    def timed(self, seconds):
        """Step repeatedly for at least `seconds`; elements per second."""
        done, t0 = 0, time.perf_counter()
        while True:
            self.step()
            done += self.n
            el = time.perf_counter() - t0
            if el >= seconds:
                return done / el, done // self.n, el

    def timed_single_thread(self, seconds, elems=1 << 18):
        """The plain oracle on one host thread, over the first `elems` of the window."""
        import oracle
        wl, a = self.wl, self.a
        n = min(elems, self.n)
        done, t0 = 0, time.perf_counter()
        while True:
            self.t += 1
            oracle.zero_step(wl.numel, wl.world, -1 if wl.rank < 0 else wl.rank, self.grads,
                             self.hw, self.hm, self.hv, self.hp, wl.lr, wl.beta1, wl.beta2,
                             wl.eps, self.t, i0=a, i1=a + n, grad_base=a, state_base=a,
                             param_base=a, grad_f32=wl.grad_f32,
                             acc_bf16=wl.acc_bf16)
            done += n
            el = time.perf_counter() - t0
            if el >= seconds:
                return done / el

    def describe(self, reps, secs):
        return (f"window [{self.a}, {self.b}) of {self.wl.name} ({self.n} elements x "
                f"{self.wl.world} ranks), stepped {reps} times in {secs:.1f} s on "
                f"{self.cores} host threads (disjoint sub-windows)")


def _cpu_oracle_sample(wl, seconds):
    s = OracleSample(wl)
    s.step()  # warm
    rate, reps, secs = s.timed(seconds)
    one = s.timed_single_thread(min(3.0, seconds))
    return {"value": rate / 1e9, "unit": "Gelem/s", "cores": s.cores, "kind": "oracle",
            "sample": s.describe(reps, secs), "single_thread_value": one / 1e9,
            "single_thread_sample": f"first {min(1 << 18, s.n)} elements of the window, "
                                    "one host thread"}


def _reference_flush_bytes(args, wl):
    """The L2 flush our arm would apply to this workload on a GB300 (L2 of 129 MiB), so
    that both arms describe the same configuration; the reference arm itself runs on
    the host and touches no GPU."""
    if args.l2 == "none" or (args.l2 == "auto"
                             and _workload_bytes(wl) >= 4 * L2_FALLBACK_BYTES):
        return None
    return 2 * L2_FALLBACK_BYTES


def run_reference(args, wl):
    """The reference arm: the CPU oracle timed on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    per_step = max(0.5, min(5.0, 60.0 / max(1, args.steps + args.warmup)))
    sample = OracleSample(wl)
    for _ in range(args.warmup):
        sample.step()
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        rate, reps, secs = sample.timed(per_step)
        vals.append(rate / 1e9)
    el = time.perf_counter() - t0
    v = statistics.median(vals)
    cb = {"value": v, "unit": "Gelem/s", "cores": sample.cores, "kind": "oracle",
          "sample": sample.describe(reps, secs) + f"; median of {args.steps} such steps"}
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "Gelem/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * el / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": _config(wl, args.unit_mode, _reference_flush_bytes(args, wl)),
        "cpu_baseline": cb,
        "e2e": {"value": v, "unit": "Gelem/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


class Refused(Exception):
    """A timed region in which a kernel gave up a bounded wait: some element of a step
    was not updated, so its time is not the time of the step and no line is printed."""


def device_state(za, dist=None, device=None) -> str:
    """'ok' if every bounded wait of the library's kernels completed since the last
    check (on every rank), else 'timeout'.  Synchronises the device."""
    bad = 0.0 if za.device_status() == za.ZERO_OK else 1.0
    if dist is not None:
        import torch
        x = torch.tensor([bad], dtype=torch.float64, device=device)
        dist.all_reduce(x, op=dist.ReduceOp.MAX)
        bad = float(x.item())
    return "ok" if bad == 0.0 else "timeout"


def require_ok(state: str, what: str) -> str:
    if state != "ok":
        raise Refused(f"{what}: a kernel gave up a bounded wait (device status {state}); "
                      "the steps did not complete and their time is not reported")
    return state


def timed_region(rep, stream, steps, t, flush=None, dist=None):
    """The timed steps t+1 .. t+steps, each bracketed by CUDA events per launch on the
    launching stream, with a barrier and a device synchronize on both sides.
    Returns (last t, events, wall seconds)."""
    import torch
    nk = len(rep.kernels)
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(nk)] for _ in range(steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(rep.dev)
    t_wall = time.perf_counter()
    for i in range(steps):
        t += 1
        if flush is not None:
            flush(i)
        rep.step(t, stream, ev[i])
    torch.cuda.synchronize(rep.dev)
    wall = time.perf_counter() - t_wall
    if dist is not None:
        dist.barrier()
    return t, ev, wall


def aggregate(ms_local: float, elems_per_rank: int, world_size: int, dist=None, device=None):
    """Whole-job throughput of N replicas: every rank's elements over the slowest rank's
    time (max over ranks).  Returns (ms_max, Gelem/s)."""
    ms = ms_local
    if dist is not None and world_size > 1:
        import torch
        x = torch.tensor([ms_local], dtype=torch.float64,
                         device=device if device is not None else "cpu")
        dist.all_reduce(x, op=dist.ReduceOp.MAX)
        ms = float(x.item())
    return ms, world_size * elems_per_rank / (ms * 1e-3) / 1e9


def _workload_bytes(wl):
    """Algorithmic bytes of one step of the workload: the step's (2N + 26) per stepped
    element, plus 4 per unit element for a ZeRO-3 unit's gather."""
    shard = -(-wl.numel // wl.world)
    return (4 * wl.numel if wl.name.startswith("unit") else 0) + _bytes_per_step(wl, shard)


def _config(wl, unit_mode="fused", flush_bytes=None):
    """The workload's description, the same for both arms: sizes, layouts, distributions,
    the algorithmic bytes per step and the L2 handling between timed steps."""
    l2 = "inputs larger than L2 (no flush)"
    if flush_bytes is not None:
        l2 = (f"L2 flushed before every timed step: a {flush_bytes >> 20} MiB write, then a "
              f"{flush_bytes >> 20} MiB read (clean lines), outside the timed launches; "
              "ms_per_step is the sum of the step's launch times")
    c = {"workload": wl.name, "numel": wl.numel, "world": wl.world,
         "rank": "all" if wl.rank < 0 else wl.rank, "grad_layout": wl.grad_layout,
         "param_layout": wl.param_layout, "grad_dist": ["normal", "student_t3"][wl.grad_dist],
         "l2": l2, "parallelism": "replicas",
         "state": "fp32 master/m/v, bf16 params",
         "gradients": "fp32" if wl.grad_f32 else "bf16",
         "reduce": "bf16-rounded sum" if wl.acc_bf16 else "fp32 sum",
         "shard": -(-wl.numel // wl.world), "bytes_per_step": _workload_bytes(wl)}
    if wl.name.startswith("unit"):
        c["unit_step"] = ("zero3_unit_step: the gather of the N shards and rank 0's step on "
                          "its shard in one call" if unit_mode == "fused" else
                          "zero3_unit_gather of the N shards, then rank 0's step on its shard")
        c["elements"] = "unit elements U per step"
    return c


def run_ours(args, wl):
    import torch
    world_size = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world_size > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        # a rank that dies fails the others' next collective after this, not after 30 min
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo",
                                timeout=datetime.timedelta(minutes=10))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    rep = Replica(wl, dev, args.unit_mode)
    stream = torch.cuda.current_stream(dev)
    # prewarm steps (state as after t = 1..prewarm), then the timed gradients
    t = 0
    for t in range(1, wl.prewarm + 1):
        rep.fill_grads(t)
        rep.step(t, stream)
    rep.fill_grads(wl.prewarm + 1)

    need = L2Flush.needed(rep.step_bytes(), dev) if args.l2 == "auto" else args.l2 == "flush"
    flush = L2Flush(dev) if need else None
    # The clock sampler starts before the warm-up steps, which run as the timed steps do
    # (with the flush) and lead straight into the timed region: a GPU left idle while
    # nvidia-smi starts lowers its clocks, and the first launch after such a pause ran
    # up to twice its usual time.
    sampler = ClockSampler(local)
    sampler.start()
    try:
        for i in range(args.warmup):
            t += 1
            if flush is not None:
                flush(i)
            rep.step(t, stream)
        torch.cuda.synchronize(dev)
        require_ok(device_state(rep.za, dist, dev), "prewarm and warm-up steps")
        t, ev, wall = timed_region(rep, stream, args.steps, t, flush, dist)
    finally:
        clocks = sampler.stop()
    status = require_ok(device_state(rep.za, dist, dev), "timed region")
    if flush is None:
        total_ms = ev[0][0][0].elapsed_time(ev[-1][-1][1])
    else:   # the flushes sit between the steps: add up the steps' own launches
        total_ms = sum(e0.elapsed_time(e1) for step in ev for e0, e1 in step)
    per_kernel = []
    for j, (name, nbytes) in enumerate(rep.kernels):
        ms = [ev[i][j][0].elapsed_time(ev[i][j][1]) for i in range(args.steps)]
        per_kernel.append({"kernel": name, "algorithmic_bytes_per_launch": nbytes,
                           "avg_launch_ms": statistics.mean(ms),
                           "median_launch_ms": statistics.median(ms),
                           "gbs": nbytes / (statistics.mean(ms) * 1e-3) / 1e9})
    elems = rep.unit_elements()
    ms_step, value = aggregate(total_ms / args.steps, elems, world_size, dist, dev)
    dom = max(per_kernel, key=lambda k: k["avg_launch_ms"])
    peak, peak_src = _peaks()
    traffic = launch_traffic(dom["kernel"], wl, rep.n)

    e2e = None
    cpu = None
    if not args.no_e2e:
        e2e = _e2e(args, rep, stream, t, dist, world_size)
        t += e2e.pop("_steps")
    if rank == 0 and world_size == 1 and not args.no_cpu_baseline:
        cpu = _cpu_oracle_sample(wl, args.cpu_seconds)

    if rank == 0:
        step_gbs = rep.step_bytes() / (ms_step * 1e-3) / 1e9
        line = {
            "metric": METRIC, "value": value, "unit": "Gelem/s", "n_gpus": world_size,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": _config(wl, rep.unit_mode, flush.nbytes if flush is not None else None),
            "launches_per_step": [k for k, _ in rep.kernels],
            "hbm_gbs": step_gbs, "hbm_frac_of_peak": step_gbs / peak,
            "roofline": {"bound": "hbm", "achieved": dom["gbs"], "peak": peak, "unit": "GB/s",
                         "frac": dom["gbs"] / peak, "traffic": traffic,
                         "peak_source": f"{peak_src} hbm_gbs (burst copy)",
                         "kernel": dom["kernel"],
                         "algorithmic_bytes_per_launch": dom["algorithmic_bytes_per_launch"],
                         "avg_launch_ms": dom["avg_launch_ms"],
                         "median_launch_ms": dom["median_launch_ms"]},
            "kernels": per_kernel,
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps * sum(2 if "+" in k else 1 for k, _ in rep.kernels),
            "clocks": clocks, "wall_s_timed": wall, "device_status": status,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def _host_available_bytes():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


def _e2e(args, rep, stream, t, dist, world_size):
    """The same step through the public API with HOST buffers.  Every step's inputs
    (the N ranks' gradients; for ZeRO-3 units also the N parameter shards) sit in
    pinned host memory and its result (the bf16 parameters of the stepped range) is
    written to pinned host memory.  The fused kernel reads the host gradients
    directly over NVLink-C2C and writes the host parameters (no staging copies),
    so every byte crosses the host link inside the timed region.  The copy-engine
    alternative (cudaMemcpyAsync in, step, out) is timed too and reported beside."""
    import torch
    wl = rep.wl
    k_steps = max(1, min(args.steps, args.e2e_steps))
    n = rep.n
    gsize = 4 if wl.grad_f32 else 2
    g_len = rep.g[0].numel()
    # every rank on this host pins its own copy: keep the total within half of what is free
    need = gsize * g_len * wl.world + 2 * rep.p.numel()
    if rep.unit:
        need += sum(2 * x.numel() for x in rep.shards)
    local_ranks = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
    avail = _host_available_bytes()
    skip = avail is not None and need * local_ranks > 0.5 * avail
    if dist is not None:   # one decision for all ranks (they meet in barriers below)
        flag = torch.tensor([1.0 if skip else 0.0], device=rep.dev)
        dist.all_reduce(flag, op=dist.ReduceOp.MAX)
        skip = flag.item() > 0
    if skip:
        return {"value": None, "unit": "Gelem/s", "h2d_bytes_per_step": gsize * n * wl.world,
                "d2h_bytes_per_step": 2 * n, "skipped": (
                    f"{local_ranks} ranks x {need / 1e9:.1f} GB of pinned host buffers exceed half "
                    f"of the host memory available"), "_steps": 0}
    hg = [torch.empty(g_len, dtype=rep.g[0].dtype, pin_memory=True) for _ in range(wl.world)]
    for k in range(wl.world):
        hg[k].copy_(rep.g[k])
    hs = None
    if rep.unit:
        hs = [torch.empty(sk.numel(), dtype=torch.int16, pin_memory=True) for sk in rep.shards]
        for hsk, sk in zip(hs, rep.shards):
            hsk.copy_(sk)
    hp = torch.empty(rep.p.numel(), dtype=torch.int16, pin_memory=True)
    torch.cuda.synchronize(rep.dev)
    in_bytes = sum(x.numel() * gsize for x in hg)
    if rep.unit:
        in_bytes = gsize * n * wl.world + sum(x.numel() * 2 for x in hs)
    elif wl.grad_layout != "shard":
        in_bytes = gsize * n * wl.world   # the kernel reads the stepped range only

    def zero_copy(tt):
        rep.step(tt, stream, grads=hg, shards=hs, param=hp)

    def copies(tt):
        for k in range(wl.world):
            rep.g[k].copy_(hg[k], non_blocking=True)
        if rep.unit:
            for sk, hsk in zip(rep.shards, hs):
                sk.copy_(hsk, non_blocking=True)
        rep.step(tt, stream)
        hp.copy_(rep.p, non_blocking=True)

    out = {}
    for name, fn in (("zero_copy", zero_copy), ("copy_engine", copies)):
        t += 1
        fn(t)  # warm-up
        torch.cuda.synchronize(rep.dev)
        if dist is not None:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(k_steps):
            t += 1
            fn(t)
        e1.record(stream)
        torch.cuda.synchronize(rep.dev)
        require_ok(device_state(rep.za, dist, rep.dev), f"e2e {name} leg")
        out[name] = aggregate(e0.elapsed_time(e1) / k_steps, rep.unit_elements(), world_size,
                              dist, rep.dev)
    ms, val = out["zero_copy"]
    return {"value": val, "unit": "Gelem/s",
            "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": 2 * n,
            "ms_per_step": ms, "steps": k_steps,
            "mode": "zero-copy: the kernel reads pinned host inputs and writes pinned host "
                    "parameters over NVLink-C2C",
            "copy_engine": {"value": out["copy_engine"][1], "ms_per_step": out["copy_engine"][0],
                            "mode": "cudaMemcpyAsync H2D, step, D2H on one stream"},
            "device_status": "ok",
            "_steps": 2 * (k_steps + 1)}


def run_zero2_buckets(args):
    """ZeRO-2 bucketed step ("Implementing ZeRO's Adam from scratch", closing note: real
    ZeRO-2 reduce-scatters bucket by bucket during the backward pass and frees each
    full-gradient bucket once it has gone out).  GPT-2-small flat vector, N = 8.  An
    emulated backward pass writes each bucket's N gradients (the seeded generator, last
    bucket first) into one of two bucket buffers on stream A; stream B steps the bucket
    (zero_adam_step_range, ZERO_GRAD_WINDOW) as soon as its event fires and hands the
    buffer back.  Gradient memory is 2 buckets instead of the full vector.

    Reported: the whole-vector step; the buckets' steps back to back (small-launch
    efficiency); the backward alone; backward then steps; the overlapped schedule."""
    import torch
    import synth
    from synth import configs as C
    import zero_partitioned_mixed_adam_gb300 as za
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl = C.GPT2
    numel, N, B = wl.numel, wl.world, args.bucket
    plan = za.zero_plan(numel, N)
    w = torch.zeros(plan.padded, dtype=torch.float32, device=dev)
    synth.fill_dev(wl.master_spec(), 0, numel, synth.OUT_F32, w.data_ptr(), 0)
    m, v = torch.zeros_like(w), torch.zeros_like(w)
    p = torch.zeros(numel, dtype=torch.int16, device=dev)
    full = [torch.zeros(plan.padded, dtype=torch.int16, device=dev) for _ in range(N)]
    for k in range(N):
        synth.fill_dev(wl.grad_spec(k, 1), 0, numel, synth.OUT_BF16, full[k].data_ptr(), 0)
    pool = [[torch.empty(B, dtype=torch.int16, device=dev) for _ in range(N)] for _ in range(2)]
    starts = list(range(0, numel, B))[::-1]
    main_s = torch.cuda.current_stream(dev)
    sb = torch.cuda.Stream(dev)
    tt = [0]

    def backward_bucket(i, b0, stream):
        n = min(B, numel - b0)
        for k in range(N):
            synth.fill_dev(wl.grad_spec(k, 1), b0, n, synth.OUT_BF16, pool[i % 2][k].data_ptr(),
                           stream.cuda_stream)

    def step_bucket(i, b0, stream):
        za.zero_adam_step_range(plan, -1, b0, b0 + B, pool[i % 2], w, m, v, p, lr=wl.lr,
                                t=tt[0], stream=stream)

    def whole():
        tt[0] += 1
        za.zero_adam_step(plan, -1, full, w, m, v, p, lr=wl.lr, t=tt[0], stream=main_s)

    def buckets_only():
        tt[0] += 1
        for i, b0 in enumerate(starts):
            step_bucket(i, b0, main_s)

    # the buckets' steps touch disjoint windows, so they need no order among themselves:
    # round-robin over two streams lets one bucket's launch start on the SMs the previous
    # one has finished with
    side = torch.cuda.Stream(dev)

    def buckets_two_streams(stream=None, other=None):
        stream = stream or main_s
        other = other or side
        tt[0] += 1
        fork = torch.cuda.Event()
        fork.record(stream)
        other.wait_event(fork)
        for i, b0 in enumerate(starts):
            step_bucket(i, b0, stream if i % 2 == 0 else other)
        join = torch.cuda.Event()
        join.record(other)
        stream.wait_event(join)

    def backward_only():
        for i, b0 in enumerate(starts):
            backward_bucket(i, b0, main_s)

    def backward_then_steps():
        tt[0] += 1
        for i, b0 in enumerate(starts):
            backward_bucket(i, b0, main_s)
            step_bucket(i, b0, main_s)

    def overlapped():
        tt[0] += 1
        free = [torch.cuda.Event(), torch.cuda.Event()]
        start = torch.cuda.Event()
        start.record(main_s)
        sb.wait_event(start)
        for e in free:
            e.record(sb)
        for i, b0 in enumerate(starts):
            ready = torch.cuda.Event()
            main_s.wait_event(free[i % 2])
            backward_bucket(i, b0, main_s)
            ready.record(main_s)
            sb.wait_event(ready)
            step_bucket(i, b0, sb)
            free[i % 2].record(sb)
        done = torch.cuda.Event()
        done.record(sb)
        main_s.wait_event(done)

    sb2 = torch.cuda.Stream(dev)

    def overlapped_two_streams():
        """As overlapped(), with bucket i stepped on side stream i % 2 (pool slot i % 2 is
        always read and released by the same stream)."""
        tt[0] += 1
        steps = [sb, sb2]
        free = [torch.cuda.Event(), torch.cuda.Event()]
        start = torch.cuda.Event()
        start.record(main_s)
        for j in (0, 1):
            steps[j].wait_event(start)
            free[j].record(steps[j])
        for i, b0 in enumerate(starts):
            ready = torch.cuda.Event()
            main_s.wait_event(free[i % 2])
            backward_bucket(i, b0, main_s)
            ready.record(main_s)
            steps[i % 2].wait_event(ready)
            step_bucket(i, b0, steps[i % 2])
            free[i % 2].record(steps[i % 2])
        for j in (0, 1):
            done = torch.cuda.Event()
            done.record(steps[j])
            main_s.wait_event(done)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(main_s)
        for _ in range(args.steps):
            fn()
        e1.record(main_s)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / args.steps

    t_whole, t_buckets = timed(whole), timed(buckets_only)
    # the same bucket steps replayed from a CUDA graph (no per-launch host work)
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for i, b0 in enumerate(starts):
                step_bucket(i, b0, cap)
    t_graph = timed(graph.replay)
    t_two = timed(buckets_two_streams)
    graph2 = torch.cuda.CUDAGraph()
    side2 = torch.cuda.Stream(dev)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph2, stream=cap):
            buckets_two_streams(cap, side2)
    t_two_graph = timed(graph2.replay)
    t_bwd, t_serial, t_over = timed(backward_only), timed(backward_then_steps), timed(overlapped)
    t_over2 = timed(overlapped_two_streams)
    status = require_ok(device_state(za), "zero2_buckets timed regions")
    peak, peak_src = _peaks()
    nbytes = (2 * N + 26) * numel
    line = {
        "metric": METRIC, "value": numel / (t_over * 1e-3) / 1e9, "unit": "Gelem/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_over,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "zero2_buckets", "numel": numel, "world": N, "bucket": B,
                   "buckets": len(starts), "gradient_memory": "2 buckets x N ranks",
                   "backward_stand_in": "seeded generator filling each bucket's N gradients",
                   "value": "parameters per overlapped backward+step pass"},
        "whole_step_ms": t_whole, "bucket_steps_ms": t_buckets,
        "small_launch_efficiency": t_whole / t_buckets,
        "bucket_steps_graph_ms": t_graph, "small_launch_efficiency_graph": t_whole / t_graph,
        "bucket_steps_two_streams_ms": t_two,
        "small_launch_efficiency_two_streams": t_whole / t_two,
        "bucket_steps_two_streams_graph_ms": t_two_graph,
        "small_launch_efficiency_two_streams_graph": t_whole / t_two_graph,
        "backward_only_ms": t_bwd, "backward_then_steps_ms": t_serial,
        "overlapped_ms": t_over, "overlapped_two_streams_ms": t_over2,
        "hidden_fraction_of_steps": (t_serial - t_over) / t_buckets,
        "roofline": {"bound": "hbm", "achieved": nbytes / (t_buckets * 1e-3) / 1e9, "peak": peak,
                     "unit": "GB/s", "frac": nbytes / (t_buckets * 1e-3) / 1e9 / peak,
                     "traffic": None, "peak_source": f"{peak_src} hbm_gbs (burst copy)",
                     "kernel": "zero_adam_step_tma_grad_kernel (per bucket: N = 8, aligned "
                               "bucket buffers and offsets)",
                     "algorithmic_bytes_per_launch": (2 * N + 26) * B,
                     "avg_launch_ms": t_buckets / len(starts)},
        "gpu_launches": len(starts) * (N + 1), "e2e": None, "cpu_baseline": None,
        "device_status": status,
    }
    print(json.dumps(line), flush=True)
    return 0


LLAMA_LAYER = [(4096, 4096)] * 4 + [(11008, 4096), (11008, 4096), (4096, 11008), (4096, 1),
               (4096, 1)]


def prefetch_pass(layers, gather, compute, main_stream, side_stream):
    """One ZeRO-3 forward pass with prefetch ("ZeRO-3 and FSDP": all-gather layer i+1's
    parameters while layer i computes).  gather(l, slot, stream) unfolds layer l into
    unit buffer `slot` (0 or 1); compute(l, slot) runs on the current (main) stream.
    The gather of layer l+1 goes to the side stream as soon as the buffer it reuses
    (layer l-1's) is free; layer l's compute waits for its own gather only."""
    import torch
    ev_g = [torch.cuda.Event() for _ in range(layers)]
    ev_c = [torch.cuda.Event() for _ in range(layers)]
    start = torch.cuda.Event()
    start.record(main_stream)
    side_stream.wait_event(start)
    gather(0, 0, side_stream)
    ev_g[0].record(side_stream)
    for li in range(layers):
        if li + 1 < layers:
            if li >= 1:
                side_stream.wait_event(ev_c[li - 1])   # slot (li+1)%2 held layer li-1
            gather(li + 1, (li + 1) % 2, side_stream)
            ev_g[li + 1].record(side_stream)
        main_stream.wait_event(ev_g[li])
        compute(li, li % 2)
        ev_c[li].record(main_stream)


def run_zero3_prefetch(args):
    """ZeRO-3 forward with prefetch: L Llama-7B-layer units, FSDP2-style row-sharded over
    N ranks.  Layer l's compute runs on the main stream while the gather of layer l+1
    runs on a side stream into the other of two unit buffers (the memory peak is two
    unfolded units).  The compute is a stand-in on the gathered weights: the layer's
    seven linear maps on T tokens (--stand-in layer: q, k, v, o, gate, up, down as bf16
    GEMMs, attention and the activation left out) or one GEMM on its first 4096x4096
    weight (--stand-in gemm).  Timed serial (gather then compute on one stream) and
    pipelined."""
    import torch
    import synth
    import zero_partitioned_mixed_adam_gb300 as za
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    L, N, T = args.layers, args.prefetch_world, args.tokens
    shard_len, U = za.rows_layout(LLAMA_LAYER, N)
    shards = [[torch.empty(shard_len, dtype=torch.int16, device=dev) for _ in range(N)]
              for _ in range(L)]
    for li in range(L):
        for r in range(N):
            synth.fill_dev(synth.Spec(seed=li, stream=7, rank=r, sigma=0.02), 0, shard_len,
                           synth.OUT_BF16, shards[li][r].data_ptr(), 0)
    full = [torch.empty(U, dtype=torch.int16, device=dev) for _ in range(2)]
    x = torch.empty(T * 4096, dtype=torch.int16, device=dev)
    synth.fill_dev(synth.Spec(seed=99, stream=8, sigma=1.0), 0, T * 4096, synth.OUT_BF16,
                   x.data_ptr(), 0)
    x = x.view(torch.bfloat16).view(T, 4096)
    y = torch.empty(T, 4096, dtype=torch.bfloat16, device=dev)
    offs, o = [], 0
    for rows, cols in LLAMA_LAYER:
        offs.append(o)
        o += rows * cols
    act = {k: torch.empty(T, 4096, dtype=torch.bfloat16, device=dev) for k in "qkva"}
    gate = torch.empty(T, 11008, dtype=torch.bfloat16, device=dev)
    up = torch.empty_like(gate)
    main_s = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(dev)

    def gather(li, slot, stream):
        za.zero3_unit_gather_rows(LLAMA_LAYER, N, shards[li], full[slot], stream=stream)

    def weight(slot, i):
        rows, cols = LLAMA_LAYER[i]
        return full[slot][offs[i]:offs[i] + rows * cols].view(torch.bfloat16).view(rows, cols)

    def compute(li, slot):
        if args.stand_in == "gemm":
            torch.matmul(x, weight(slot, 0).t(), out=y)
            return
        for i, k in enumerate("qkv"):
            torch.matmul(x, weight(slot, i).t(), out=act[k])
        torch.matmul(act["v"], weight(slot, 3).t(), out=act["a"])   # o: attention left out
        torch.matmul(act["a"], weight(slot, 4).t(), out=gate)
        torch.matmul(act["a"], weight(slot, 5).t(), out=up)
        gate.mul_(up)                                               # activation left out
        torch.matmul(gate, weight(slot, 6).t(), out=y)

    def serial():
        for li in range(L):
            gather(li, 0, main_s)
            compute(li, 0)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(main_s)
        for _ in range(args.steps):
            fn()
        e1.record(main_s)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / args.steps

    t_g = timed(lambda: [gather(li, li % 2, main_s) for li in range(L)])
    t_c = timed(lambda: [compute(li, li % 2) for li in range(L)])
    t_ser = timed(serial)
    t_pipe = timed(lambda: prefetch_pass(L, gather, compute, main_s, side))
    status = require_ok(device_state(za), "zero3_prefetch timed regions")
    peak, peak_src = _peaks()
    g_gbs = 4 * U * L / (t_g * 1e-3) / 1e9
    # the library copies on the TMA engine when every tensor offset and row block is a
    # multiple of 8 elements and every buffer is 16-byte aligned (this layout, whole buffers)
    o, ok = 0, True
    for rows, cols in LLAMA_LAYER:
        ok = ok and o % 8 == 0 and (-(-rows // N) * cols) % 8 == 0
        o += rows * cols
    ok = ok and all(x.data_ptr() % 16 == 0 for x in full + [t for layer in shards for t in layer])
    kname = "zero3_unit_gather_rows_tma_kernel" if ok else "zero3_unit_gather_rows_kernel"
    rec = (_traffic_record(os.path.join(ROOT, "zero_partitioned_mixed_adam_gb300", "csrc",
                                        "unit_gather.cu")) or {}).get(f"{kname}/N{N}")
    traffic = rec["dram_bytes_per_element"] * U if rec else None
    line = {
        "metric": METRIC, "value": L * U / (t_pipe * 1e-3) / 1e9, "unit": "Gelem/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_pipe,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "zero3_prefetch", "layers": L, "world": N,
                   "unit": "Llama-7B layer, 202,383,360 elements, FSDP2-style row shards",
                   "tokens": T, "stand_in_compute": (
                       "one bf16 GEMM [T,4096]x[4096,4096]^T (cuBLAS)" if args.stand_in == "gemm"
                       else "the layer's seven linear maps on T tokens with its gathered "
                            "weights (bf16 GEMMs, cuBLAS; attention and activation left out)"),
                   "buffers": "two unfolded units (double buffering)",
                   "elements": "unit elements gathered per pass"},
        "serial_ms": t_ser, "pipelined_ms": t_pipe, "gathers_only_ms": t_g,
        "computes_only_ms": t_c,
        "hidden_fraction_of_shorter": (t_ser - t_pipe) / min(t_g, t_c),
        "roofline": {"bound": "hbm", "achieved": g_gbs, "peak": peak, "unit": "GB/s",
                     "frac": g_gbs / peak, "traffic": traffic,
                     "peak_source": f"{peak_src} hbm_gbs (burst copy)",
                     "kernel": kname,
                     "algorithmic_bytes_per_launch": 4 * U, "avg_launch_ms": t_g / L},
        "gpu_launches": L, "e2e": None, "cpu_baseline": None, "device_status": status,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1, help="GPUs (one process each under torchrun)")
    ap.add_argument("--steps", type=int, default=50, help="timed steps")
    ap.add_argument("--warmup", type=int, default=5, help="untimed steps first (>= 3)")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours",
                    help="reference: the CPU oracle on the host cores")
    ap.add_argument("--workload", default="1p3b",
                    help="1p3b | gpt2 | 7b_rank3 | 7b_rank3_prewarm | tiny | unit:U:N | "
                         "shard:U:N | zero2_buckets | zero3_prefetch")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer run")
    ap.add_argument("--e2e-steps", type=int, default=5, help="steps of the host-buffer run")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="seconds of oracle timing on all host cores")
    ap.add_argument("--bucket", type=int, default=1 << 24, help="zero2_buckets: elements")
    ap.add_argument("--layers", type=int, default=8, help="zero3_prefetch: units per pass")
    ap.add_argument("--prefetch-world", type=int, default=8, help="zero3_prefetch: ranks")
    ap.add_argument("--tokens", type=int, default=4096, help="zero3_prefetch: GEMM rows")
    ap.add_argument("--stand-in", choices=("layer", "gemm"), default="layer",
                    help="zero3_prefetch: each layer's compute, its seven linear maps on the "
                         "tokens (layer) or one 4096x4096 GEMM (gemm)")
    ap.add_argument("--grad-variant", choices=("bf16", "f32", "bf16sum"), default="bf16",
                    help="gradients in bf16 (the method), fp32 (the page's runnable demo), or "
                         "bf16 with the sum over ranks rounded to bf16 after every addition")
    ap.add_argument("--l2", choices=("auto", "flush", "none"), default="auto",
                    help="flush the L2 before every timed step: auto = when a step moves less "
                         "than four L2 sizes")
    ap.add_argument("--unit-mode", choices=("fused", "separate"), default="fused",
                    help="unit workloads: one zero3_unit_step call, or the gather and the "
                         "step as two calls")
    ap.add_argument("--numel", type=int, default=0,
                    help="override the workload's parameter count (smaller profiling cases)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    try:
        if args.workload == "zero3_prefetch":
            return run_zero3_prefetch(args)
        if args.workload == "zero2_buckets":
            return run_zero2_buckets(args)
        wl = _workload(args.workload)
        import dataclasses
        if args.numel:
            wl = dataclasses.replace(wl, numel=args.numel, name=f"{wl.name}@numel={args.numel}")
        if args.grad_variant != "bf16":
            wl = dataclasses.replace(wl, grad_f32=args.grad_variant == "f32",
                                     acc_bf16=args.grad_variant == "bf16sum",
                                     name=f"{wl.name}+{args.grad_variant}")
        if args.impl == "reference":
            return run_reference(args, wl)
        return run_ours(args, wl)
    except Refused as e:
        print(f"bench.py: refused: {e}", file=sys.stderr, flush=True)
        return 3


if __name__ == "__main__":
    sys.exit(main())
