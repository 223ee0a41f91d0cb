"""The ZeroAdam object on the page's own demo: the MLP Linear(64,256)-GELU-Linear(256,10),
4 ranks each with a quarter of a 32-example batch, 3 steps.  The ranks' backward
passes are a stand-in (torch autograd on a float copy of the current bf16
parameters); their gradients, cast to bf16, go into each rank's gradient buffer.
The fp32 state must equal the oracle's on the same gradient bytes (bit for bit),
and stay close to single-process fp32 torch.optim.Adam on the full batch: the
page's demo is fp32 throughout and meets 1e-5; with bf16 forward weights and
bf16 gradients (~0.4 % relative) the moments' ratios move the updates by about
lr * 0.4 %, and a gradient whose sign flips moves one element by up to 2 lr."""
import numpy as np
import pytest
import torch

import oracle
from conftest import cuda_available
import gpu_util as gu

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]

from zero_partitioned_mixed_adam_gb300.optim import ZeroAdam  # noqa: E402


def _model():
    torch.manual_seed(0)
    return torch.nn.Sequential(torch.nn.Linear(64, 256), torch.nn.GELU(), torch.nn.Linear(256, 10))


def test_zero_adam_object_on_the_demo_mlp():
    world, lr = 4, 1e-2
    torch.manual_seed(123)
    X, Y = torch.randn(32, 64), torch.randint(0, 10, (32,))
    ref = _model()
    model = _model().cuda()               # fp32 weights: the master starts from them exactly
    opt = ZeroAdam(model.parameters(), lr=lr, world=world)
    assert all(p.dtype == torch.bfloat16 for p in model.parameters())
    assert opt.numel == 19_210 and opt.shard == 4_803
    assert opt.state_bytes() == 57_636
    opt_ref = torch.optim.Adam(ref.parameters(), lr=lr, foreach=False)
    loss_fn = torch.nn.CrossEntropyLoss()
    numel, P = opt.numel, opt.plan.padded
    hw = np.zeros(P, np.float32)
    hw[:numel] = gu.to_host_f32(opt.master)[:numel]
    hm, hv, hp = np.zeros(P, np.float32), np.zeros(P, np.float32), np.zeros(numel, np.uint16)
    for t in range(1, 4):
        opt.zero_grad()
        for k in range(world):
            local = slice(k * 32 // world, (k + 1) * 32 // world)
            shadow = _model()
            with torch.no_grad():
                for a, b in zip(shadow.parameters(), model.parameters()):
                    a.copy_(b.float().cpu())
            # each rank's loss is the mean over its quarter; the sum over ranks
            # divided by N is the full-batch mean's gradient
            loss_fn(shadow(X[local]), Y[local]).backward()
            for g, p in zip(opt.grads_of(k), shadow.parameters()):
                g.copy_(p.grad.to(torch.bfloat16))
        opt.step()
        hg = [gu.to_host_u16(g) for g in opt.grads]
        oracle.zero_step(numel, world, -1, hg, hw, hm, hv, hp, lr, 0.9, 0.999, 1e-8, t)
        opt_ref.zero_grad()
        loss_fn(ref(X), Y).backward()
        opt_ref.step()
    torch.cuda.synchronize()
    gu.assert_f32_close(gu.to_host_f32(opt.master)[:numel], hw[:numel], "ZeroAdam master")
    gu.assert_f32_close(gu.to_host_f32(opt.m)[:numel], hm[:numel], "ZeroAdam m")
    gu.assert_bf16_close(gu.to_host_u16(opt.flat_params), hp, "ZeroAdam params")
    # the parameters are views into the all-gathered flat buffer
    flat = torch.cat([p.detach().reshape(-1) for p in model.parameters()])
    assert torch.equal(flat, opt.flat_params)
    w_ref = torch.cat([p.detach().reshape(-1) for p in ref.parameters()]).numpy()
    diff = np.abs(gu.to_host_f32(opt.master)[:numel] - w_ref)
    assert np.median(diff) < 1e-4
    assert diff.max() <= 3 * 2 * lr


def test_pointer_array_and_a_replaced_gradient_buffer():
    """The same step through a list of gradient buffers and through a PointerArray of them
    gives the same bits; ZeroAdam, which keeps a PointerArray of its buffers, steps on a
    gradient buffer that replaced one of them."""
    import zero_partitioned_mixed_adam_gb300 as za
    world = 4
    opts = []
    for replace in (False, True):
        model = _model().cuda()
        opt = ZeroAdam(model.parameters(), lr=1e-2, world=world)
        for k in range(world):
            g = opt.grads[k]
            g.copy_(torch.randn(g.numel(), generator=torch.Generator().manual_seed(k)).to(
                torch.bfloat16))
        x = torch.randn(opt.grads[2].numel(), generator=torch.Generator().manual_seed(99)).to(
            device=opt.grads[2].device, dtype=torch.bfloat16)
        if replace:   # rank 2's gradients in a new buffer; the old one keeps other values
            opt.grads[2] = x
        else:
            opt.grads[2].copy_(x)
        opt.step(check=True)
        opts.append(opt)
    torch.cuda.synchronize()
    for name in ("master", "m", "v", "flat_params"):   # bit for bit
        assert torch.equal(getattr(opts[0], name).view(torch.int16),
                           getattr(opts[1], name).view(torch.int16)), name
    # the raw call: a list and a PointerArray of the same buffers
    o = opts[0]
    outs = []
    for grads in (list(o.grads), za.pointer_array(o.grads)):
        w, m, v = o.master.clone(), o.m.clone(), o.v.clone()
        p = torch.empty_like(o.flat_params)
        za.zero_adam_step(o.plan, za.ZERO_ALL_RANKS, grads, w, m, v, p, lr=1e-2, t=2)
        outs.append((w, m, v, p))
    za.check_device("pointer array step")
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
