"""The device input generator reproduces the host generator bit for bit, so the
oracle (host inputs) and the CUDA path (device inputs) see the same bytes."""
import numpy as np
import pytest
import torch

import synth
from conftest import cuda_available

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]


@pytest.mark.parametrize("spec", [
    synth.Spec(seed=0, stream=1, rank=3, step=2, sigma=1e-3),
    synth.Spec(seed=0, stream=1, rank=0, step=1, sigma=1e-3, zero_frac=0.1),
    synth.Spec(seed=5, stream=1, rank=15, step=6, dist=synth.STUDENT_T3, sigma=1e-3,
               outlier_rate=1e-3, outlier_value=100.0),
    synth.Spec(seed=0, stream=2, sigma=0.02),
])
@pytest.mark.parametrize("kind", [synth.OUT_F32, synth.OUT_BF16])
def test_device_generator_equals_host(spec, kind):
    for offset, n in ((0, 1), (7, 1000), (2**33 + 5, 4099), (123456, 1 << 20)):
        dt = torch.float32 if kind == synth.OUT_F32 else torch.int16
        t = torch.empty(n, dtype=dt, device="cuda")
        synth.fill_dev(spec, offset, n, kind, t.data_ptr(), 0)
        torch.cuda.synchronize()
        dev = t.cpu().numpy()
        if kind == synth.OUT_BF16:
            dev = dev.view(np.uint16)
        host = synth.fill_host(spec, offset, n, kind)
        assert (dev.view(np.uint8) == host.view(np.uint8)).all(), (offset, n)
