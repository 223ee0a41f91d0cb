"""bench.py refuses a timed region in which a kernel gave up a bounded wait.

The library's test hook makes the TMA-staged kernels' producers issue no copies, so
every consumer wait runs out after its one-second limit and the step's outputs are
not written: such a step is fast and wrong, and its time must never become a bench
line.  The bench's own timed-region helper runs one step of a small all-ranks N = 16
workload with the hook on; the device state that follows must be 'timeout' and
require_ok must refuse it.  A second region without the hook passes."""
import pytest
import torch

from synth import configs as C
from conftest import cuda_available

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]

import bench  # noqa: E402
import zero_partitioned_mixed_adam_gb300 as za  # noqa: E402


def test_timed_region_with_a_given_up_wait_is_refused():
    dev = torch.device("cuda", 0)
    wl = C.StepWorkload("probe_n16", numel=1_000_003, world=16)
    rep = bench.Replica(wl, dev)
    assert rep.step_kernel_name() == "zero_adam_step_tma_grad_kernel"
    stream = torch.cuda.current_stream(dev)
    rep.fill_grads(1)
    assert bench.device_state(za) == "ok"
    prev = za.test_withhold_copies(True)
    try:
        t, ev, wall = bench.timed_region(rep, stream, 1, 0)
    finally:
        za.test_withhold_copies(prev)
    assert t == 1 and wall > 0.5          # the consumers waited out their limit
    state = bench.device_state(za)
    assert state == "timeout"
    with pytest.raises(bench.Refused):
        bench.require_ok(state, "timed region")
    # the same helper without the hook: the region completes and passes
    t, ev, wall = bench.timed_region(rep, stream, 2, t)
    assert bench.require_ok(bench.device_state(za), "timed region") == "ok"
    assert ev[0][0][0].elapsed_time(ev[-1][-1][1]) > 0
