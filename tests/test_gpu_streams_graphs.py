"""The entry points keep no state, allocate nothing and never synchronise, so calls on
different streams may run concurrently, and a sequence of calls can be captured into a
CUDA graph and replayed; both give the bits of plain sequential calls."""
import pytest
import torch

import synth
from synth import configs as C
from conftest import cuda_available

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]

import zero_partitioned_mixed_adam_gb300 as za  # noqa: E402


def _setup(numel, world, seed=2):
    plan = za.zero_plan(numel, world)
    g = [torch.zeros(plan.padded, dtype=torch.int16, device="cuda") for _ in range(world)]
    for k in range(world):
        synth.fill_dev(synth.Spec(seed=seed, stream=C.STREAM_GRAD, rank=k, step=1, sigma=1e-3),
                       0, numel, synth.OUT_BF16, g[k].data_ptr(), 0)
    w = torch.zeros(plan.padded, dtype=torch.float32, device="cuda")
    synth.fill_dev(synth.Spec(seed=seed, stream=C.STREAM_MASTER, sigma=0.02), 0, numel,
                   synth.OUT_F32, w.data_ptr(), 0)
    return plan, g, w


def _same(xs, ys):
    return all(torch.equal(x.view(torch.int32) if x.dtype == torch.float32 else x,
                           y.view(torch.int32) if y.dtype == torch.float32 else y)
               for x, y in zip(xs, ys))


@pytest.mark.parametrize("world", [8, 16])
def test_ranks_on_concurrent_streams(world):
    """Every rank's single-rank step on its own stream, all in flight together."""
    numel = 4_000_003
    plan, g, w0 = _setup(numel, world)
    S = plan.shard
    ref = [w0.clone(), torch.zeros_like(w0), torch.zeros_like(w0),
           torch.zeros(numel, dtype=torch.int16, device="cuda")]
    za.zero_adam_step(plan, -1, g, *ref, lr=1e-3, t=1)
    # per-rank state views of a second copy (a rank's shard of master/m/v is contiguous)
    w, m, v = w0.clone(), torch.zeros_like(w0), torch.zeros_like(w0)
    p = torch.zeros(numel, dtype=torch.int16, device="cuda")
    streams = [torch.cuda.Stream() for _ in range(world)]
    torch.cuda.synchronize()
    for r in range(world):
        with torch.cuda.stream(streams[r]):
            za.zero_adam_step(plan, r, g, w[r * S:(r + 1) * S], m[r * S:(r + 1) * S],
                              v[r * S:(r + 1) * S], p, lr=1e-3, t=1, stream=streams[r])
    torch.cuda.synchronize()
    assert _same((w, m, v, p), ref)


@pytest.mark.parametrize("world", [4, 8, 16])
def test_bucket_sequence_captured_in_a_cuda_graph(world):
    """Bucket steps (register-staged kernel at N = 4, TMA-staged at N = 8 and 16) and a
    unit gather, captured together and replayed."""
    numel, bucket = 3_000_017, 1 << 18
    plan, g, w0 = _setup(numel, world)
    starts = list(range(0, numel, bucket))[::-1]
    uplan = za.zero_plan(1_000_003, world)
    shards = [torch.full((uplan.shard,), k, dtype=torch.int16, device="cuda")
              for k in range(world)]
    full = torch.zeros(1_000_003, dtype=torch.int16, device="cuda")

    def run(state, t, stream=None):
        for b0 in starts:
            za.zero_adam_step_range(plan, -1, b0, b0 + bucket, g, *state, lr=1e-3, t=t,
                                    grad_layout=za.ZERO_GRAD_FULL, stream=stream)
        za.zero3_unit_gather(uplan, shards, full, stream=stream)

    graphed = [w0.clone(), torch.zeros_like(w0), torch.zeros_like(w0),
               torch.zeros(numel, dtype=torch.int16, device="cuda")]
    run(graphed, 1)                       # first calls (per-device set-up) outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            run(graphed, 2)               # t is baked into the captured launches
    graph.replay()
    torch.cuda.synchronize()
    check = [x.clone() for x in graphed]
    eager2 = [w0.clone(), torch.zeros_like(w0), torch.zeros_like(w0),
              torch.zeros(numel, dtype=torch.int16, device="cuda")]
    for t in (1, 2):
        run(eager2, t)
    torch.cuda.synchronize()
    assert _same(check, eager2)
    assert torch.equal(full, torch.cat(shards)[:1_000_003])
    assert za.device_status() == 0


@pytest.mark.parametrize("world", [4, 8, 64])
def test_unit_step_captured_in_a_cuda_graph(world):
    """A small ZeRO-3 unit's gather + step (one launch at these sizes) captured once, with
    the buffers passed as pointer arrays, and replayed twice: the same bits as the same
    calls made eagerly (a loop over small units replays a graph instead of paying the host
    marshalling and the launch for every unit)."""
    U = 1 << 20
    plan = za.zero_plan(U, world)
    S = plan.shard
    shards = [torch.full((S,), 100 + k, dtype=torch.int16, device="cuda") for k in range(world)]
    gen = torch.Generator(device="cuda").manual_seed(world)
    grads = [(torch.randn(S, generator=gen, device="cuda") * 1e-3).to(torch.bfloat16)
             .view(torch.int16) for _ in range(world)]
    w0 = torch.randn(S, generator=gen, device="cuda") * 0.02
    sp, gp = za.pointer_array(shards), za.pointer_array(grads)

    def fresh():
        return [torch.zeros(U, dtype=torch.int16, device="cuda"), w0.clone(),
                torch.zeros_like(w0), torch.zeros_like(w0),
                torch.zeros(S, dtype=torch.int16, device="cuda")]

    def run(bufs, t, s_arg, g_arg, stream=None):
        full, w, m, v, p = bufs
        za.zero3_unit_step(plan, 1, s_arg, full, g_arg, w, m, v, p, lr=1e-3, t=t,
                           grad_layout=za.ZERO_GRAD_SHARD, param_layout=za.ZERO_PARAM_SHARD,
                           stream=stream)

    graphed = fresh()
    run(graphed, 1, sp, gp)               # per-device set-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            run(graphed, 2, sp, gp)       # t = 2 is baked into the captured launch
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    eager = fresh()
    for t in (1, 2, 2):
        run(eager, t, list(shards), list(grads))
    torch.cuda.synchronize()
    assert _same(graphed, eager)
    assert torch.equal(graphed[0], torch.cat(shards)[:U])
    assert za.device_status() == 0
