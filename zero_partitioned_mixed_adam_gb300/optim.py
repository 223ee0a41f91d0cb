"""ZeroAdam: the page's optimizer object over the C ABI, N ranks emulated on one GPU.

Same surface as the class in "ZeRO and FSDP" -> "Implementing ZeRO's Adam from
scratch": ZeroAdam(params, lr, betas=(0.9, 0.999), eps=1e-8), step(),
zero_grad(), state_bytes().  The flat layout is the page's (numel, shard =
ceil(numel/world), zero-padded tail); the differences are GB300-first:

- the parameters become views into one flat bf16 buffer, which is where the
  kernel's all-gather writes, so there is no unflatten copy;
- each emulated rank k owns a flat bf16 gradient buffer (grads_of(k) gives
  per-parameter views of it, for that rank's backward pass to fill);
- the fp32 master weights, m and v of all ranks live in three flat buffers;
- step() is one zero_adam_step launch on the current stream (no collectives:
  the ranks are buffers in this GPU's memory).

This module only allocates (through PyTorch) and marshals; the arithmetic runs
in libzeroadam.so.
"""
from __future__ import annotations

import torch

from . import ZERO_ALL_RANKS, check_device, pointer_array, zero_adam_step, zero_plan


class ZeroAdam:
    def __init__(self, params, lr, betas=(0.9, 0.999), eps=1e-8, world=1):
        self.params = list(params)
        self.lr, self.betas, self.eps, self.t = lr, betas, eps, 0
        self.world = world
        dev = self.params[0].device
        if dev.type != "cuda":
            raise ValueError("ZeroAdam keeps its state in GPU memory: give it CUDA parameters")
        self.numel = sum(p.numel() for p in self.params)
        self.plan = zero_plan(self.numel, world)
        self.shard = self.plan.shard
        padded = self.plan.padded
        # fp32 master weights of every rank's shard (the page keeps only the own
        # slice per process; here all N slices live side by side), moments at zero
        self.master = torch.zeros(padded, dtype=torch.float32, device=dev)
        self.m = torch.zeros_like(self.master)
        self.v = torch.zeros_like(self.master)
        self.flat_params = torch.empty(self.numel, dtype=torch.bfloat16, device=dev)
        self.grads = [torch.zeros(padded, dtype=torch.bfloat16, device=dev) for _ in range(world)]
        self._grad_ptrs = pointer_array(self.grads)
        off = 0
        with torch.no_grad():
            for p in self.params:
                n = p.numel()
                self.master[off:off + n] = p.detach().reshape(-1).float()
                view = self.flat_params[off:off + n].view(p.shape)
                view.copy_(p.detach())
                p.data = view
                off += n

    def grads_of(self, k):
        """Per-parameter views into emulated rank k's flat bf16 gradient buffer."""
        out, off = [], 0
        for p in self.params:
            out.append(self.grads[k][off:off + p.numel()].view(p.shape))
            off += p.numel()
        return out

    def step(self, stream=None, check=False):
        """One ZeRO-2 step of every rank: reduce-scatter + average, Adam, all-gather.

        With check=True the call waits for the device and raises ZeroError
        (ZERO_E_TIMEOUT) if a kernel gave up a bounded wait, i.e. if some element
        of the step was not updated."""
        self.t += 1
        b1, b2 = self.betas
        if any(a is not b for a, b in zip(self.grads, self._grad_ptrs.buffers)):
            self._grad_ptrs = pointer_array(self.grads)   # a gradient buffer was replaced
        zero_adam_step(self.plan, ZERO_ALL_RANKS, self._grad_ptrs, self.master, self.m, self.v,
                       self.flat_params, lr=self.lr, beta1=b1, beta2=b2, eps=self.eps, t=self.t,
                       stream=stream)
        if check:
            check_device("ZeroAdam.step")

    def zero_grad(self):
        for g in self.grads:
            g.zero_()

    def state_bytes(self):
        """fp32 master + m + v bytes one rank holds (12 x shard)."""
        return 3 * 4 * self.shard
