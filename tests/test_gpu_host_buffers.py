"""The end-to-end path with host buffers: gradients in pinned host memory and the
bf16 parameters written to pinned host memory, read and written by the kernels
directly (NVLink-C2C on GB300).  The result must equal the all-device step bit
for bit, on the register-staged kernel (N = 4) and the TMA-staged one (N = 8, 16
and 64: gradients staged in rank groups of 8 and of 32)."""
import pytest
import torch

import synth
from synth import configs as C
from conftest import cuda_available

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]

import zero_partitioned_mixed_adam_gb300 as za  # noqa: E402


@pytest.mark.parametrize("world", [4, 8, 16, 64])
def test_host_resident_gradients_and_parameters(world):
    numel = 3_000_017
    plan = za.zero_plan(numel, world)
    gd = [torch.zeros(plan.padded, dtype=torch.int16, device="cuda") for _ in range(world)]
    for k in range(world):
        synth.fill_dev(synth.Spec(seed=1, stream=C.STREAM_GRAD, rank=k, step=1, sigma=1e-3), 0,
                       numel, synth.OUT_BF16, gd[k].data_ptr(), 0)
    gh = [torch.empty(plan.padded, dtype=torch.int16, pin_memory=True) for _ in range(world)]
    for h, d in zip(gh, gd):
        h.copy_(d)
    w0 = torch.zeros(plan.padded, dtype=torch.float32, device="cuda")
    synth.fill_dev(synth.Spec(seed=1, stream=C.STREAM_MASTER, sigma=0.02), 0, numel,
                   synth.OUT_F32, w0.data_ptr(), 0)
    outs = []
    for grads, param in ((gd, torch.zeros(numel, dtype=torch.int16, device="cuda")),
                         (gh, torch.zeros(numel, dtype=torch.int16, pin_memory=True))):
        w, m, v = w0.clone(), torch.zeros_like(w0), torch.zeros_like(w0)
        for t in (1, 2):
            za.zero_adam_step(plan, -1, grads, w, m, v, param, lr=1e-3, t=t)
        torch.cuda.synchronize()
        outs.append((w, m, v, param.cpu()))
    for a, b in zip(outs[0][:3], outs[1][:3]):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.equal(outs[0][3].cpu(), outs[1][3])
    assert za.device_status() == 0
