"""The bounded waits of the TMA kernels (the staged step kernels and the unit gather's
copy), driven to run out without faulting or hanging the GPU: the library's test hook
makes the producers issue no copies, so every wait on a stage gives up after its limit
(one second of the GPU's global timer).  The launch must end, write nothing, and leave
ZERO_E_TIMEOUT in the device status word; the word must clear on reading, and the next
normal call on the same context must give the same bits as one that never saw the hook."""
import time

import pytest
import torch

import synth
from synth import configs as C
from conftest import cuda_available

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]

import zero_partitioned_mixed_adam_gb300 as za  # noqa: E402

E_TIMEOUT = {v: k for k, v in za.ERRORS.items()}["ZERO_E_TIMEOUT"]


def _setup(numel, world):
    plan = za.zero_plan(numel, world)
    g = [torch.zeros(plan.padded, dtype=torch.int16, device="cuda") for _ in range(world)]
    for k in range(world):
        synth.fill_dev(synth.Spec(seed=5, stream=C.STREAM_GRAD, rank=k, step=1, sigma=1e-3), 0,
                       numel, synth.OUT_BF16, g[k].data_ptr(), 0)
    w0 = torch.zeros(plan.padded, dtype=torch.float32, device="cuda")
    synth.fill_dev(synth.Spec(seed=5, stream=C.STREAM_MASTER, sigma=0.02), 0, numel,
                   synth.OUT_F32, w0.data_ptr(), 0)
    return plan, g, w0


def _fresh(w0, numel):
    return [w0.clone(), torch.zeros_like(w0), torch.zeros_like(w0),
            torch.full((numel,), 0x1234, dtype=torch.int16, device="cuda")]


def _bits(x):
    return x.view(torch.int32) if x.dtype == torch.float32 else x


@pytest.mark.parametrize("world", [5, 8, 16, 64, 100])
def test_withheld_copies_time_out_and_the_context_survives(world):
    numel = 1_000_003
    plan, g, w0 = _setup(numel, world)
    state = _fresh(w0, numel)
    torch.cuda.synchronize()
    assert za.device_status() == za.ZERO_OK
    prev = za.test_withhold_copies(True)
    try:
        t0 = time.perf_counter()
        za.zero_adam_step(plan, -1, g, *state, lr=1e-3, t=1)   # launches; nothing arrives
        torch.cuda.synchronize()
        waited = time.perf_counter() - t0
    finally:
        za.test_withhold_copies(prev)
    assert za.device_status() == E_TIMEOUT
    assert 0.5 < waited < 60, waited        # about the one-second limit, and it ended
    assert za.device_status() == za.ZERO_OK    # reading cleared the word
    untouched = _fresh(w0, numel)
    for a, b in zip(state, untouched):
        assert torch.equal(_bits(a), _bits(b)), "a withheld step wrote an output"
    # the same context steps normally, with the bits of a step that never saw the hook
    za.zero_adam_step(plan, -1, g, *state, lr=1e-3, t=1)
    ref = _fresh(w0, numel)
    za.zero_adam_step(plan, -1, g, *ref, lr=1e-3, t=1)
    torch.cuda.synchronize()
    for a, b in zip(state, ref):
        assert torch.equal(_bits(a), _bits(b))
    assert not torch.equal(state[0], w0)
    assert za.device_status() == za.ZERO_OK


@pytest.mark.parametrize("world", [8, 16])
def test_timeout_on_a_side_stream_is_seen_without_a_torch_synchronize(world):
    """The step runs on a non-blocking torch stream and device_status() is called
    straight after the launch returns: the call itself must wait for the kernel
    (it synchronises the device) and report its timeout."""
    numel = 1_000_003
    plan, g, w0 = _setup(numel, world)
    state = _fresh(w0, numel)
    torch.cuda.synchronize()
    assert za.device_status() == za.ZERO_OK
    side = torch.cuda.Stream()
    prev = za.test_withhold_copies(True)
    try:
        za.zero_adam_step(plan, -1, g, *state, lr=1e-3, t=1, stream=side)
        status = za.device_status()     # no torch synchronize before it
    finally:
        za.test_withhold_copies(prev)
    assert status == E_TIMEOUT
    assert za.device_status() == za.ZERO_OK


def test_zero_adam_check_raises_on_a_given_up_wait():
    from zero_partitioned_mixed_adam_gb300.optim import ZeroAdam
    params = [torch.nn.Parameter(torch.randn(1 << 16, device="cuda")) for _ in range(4)]
    opt = ZeroAdam(params, lr=1e-3, world=16)
    opt.step(check=True)                  # completes: no error
    prev = za.test_withhold_copies(True)
    try:
        with pytest.raises(za.ZeroError) as e:
            opt.step(check=True)
    finally:
        za.test_withhold_copies(prev)
    assert e.value.code == "ZERO_E_TIMEOUT"
    opt.step(check=True)


def test_hook_leaves_the_register_staged_kernel_alone():
    """N = 4 runs the register-staged kernel, which has no waits: the hook changes
    nothing there."""
    numel, world = 300_007, 4
    plan, g, w0 = _setup(numel, world)
    a, b = _fresh(w0, numel), _fresh(w0, numel)
    prev = za.test_withhold_copies(True)
    try:
        za.zero_adam_step(plan, -1, g, *a, lr=1e-3, t=1)
        torch.cuda.synchronize()
    finally:
        za.test_withhold_copies(prev)
    za.zero_adam_step(plan, -1, g, *b, lr=1e-3, t=1)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(_bits(x), _bits(y))
    assert za.device_status() == za.ZERO_OK


def test_withheld_gather_times_out_and_the_context_survives():
    U, N = 1_048_573, 8          # shard 131,072: the TMA copy, with a 5-element tail
    plan = za.zero_plan(U, N)
    assert plan.shard % 8 == 0
    shards = [torch.full((plan.shard,), k + 1, dtype=torch.int16, device="cuda") for k in range(N)]
    full = torch.full((U,), -7, dtype=torch.int16, device="cuda")
    torch.cuda.synchronize()
    assert za.device_status() == za.ZERO_OK
    prev = za.test_withhold_copies(True)
    try:
        t0 = time.perf_counter()
        za.zero3_unit_gather(plan, shards, full)
        torch.cuda.synchronize()
        waited = time.perf_counter() - t0
    finally:
        za.test_withhold_copies(prev)
    assert za.device_status() == E_TIMEOUT
    assert 0.5 < waited < 60, waited
    assert bool((full == -7).all()), "a withheld gather wrote the unit"
    za.zero3_unit_gather(plan, shards, full)
    torch.cuda.synchronize()
    assert torch.equal(full, torch.cat(shards)[:U])
    assert za.device_status() == za.ZERO_OK


def test_withheld_row_gather_times_out_and_the_context_survives():
    shapes, world = [(1001, 8), (77, 16), (9, 8), (37, 4)], 4   # the TMA row copy
    shard_len, total = za.rows_layout(shapes, world)
    shards = [torch.full((shard_len,), k + 1, dtype=torch.int16, device="cuda")
              for k in range(world)]
    full = torch.full((total,), -7, dtype=torch.int16, device="cuda")
    torch.cuda.synchronize()
    assert za.device_status() == za.ZERO_OK
    prev = za.test_withhold_copies(True)
    try:
        za.zero3_unit_gather_rows(shapes, world, shards, full)
        torch.cuda.synchronize()
    finally:
        za.test_withhold_copies(prev)
    assert za.device_status() == E_TIMEOUT
    assert bool((full == -7).all()), "a withheld row gather wrote the unit"
    za.zero3_unit_gather_rows(shapes, world, shards, full)
    torch.cuda.synchronize()
    assert za.device_status() == za.ZERO_OK
    # every element of tensor i's rows [r*R, (r+1)*R) comes from rank r
    off = 0
    for rows, cols in shapes:
        R = -(-rows // world)
        t = full[off:off + rows * cols].view(rows, cols)
        for r in range(world):
            blk = t[r * R:min((r + 1) * R, rows)]
            assert bool((blk == r + 1).all())
        off += rows * cols
