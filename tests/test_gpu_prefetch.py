"""The ZeRO-3 prefetch schedule (bench.prefetch_pass): with two unit buffers and the
next layer's gather on a side stream, every layer's compute must see exactly its
own gathered unit."""
import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import cuda_available

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")]

import bench  # noqa: E402
import zero_partitioned_mixed_adam_gb300 as za  # noqa: E402


@pytest.mark.parametrize("layers,world", [(1, 4), (2, 8), (7, 3), (12, 64)])
def test_prefetch_pass_gives_each_layer_its_own_unit(layers, world):
    shapes = [(257, 33), (64, 64), (5, 1)]
    shard_len, total = za.rows_layout(shapes, world)
    host = [[synth.fill_host(synth.Spec(seed=li, stream=7, rank=r, sigma=0.02), 0, shard_len,
                             synth.OUT_BF16) for r in range(world)] for li in range(layers)]
    shards = [[torch.from_numpy(h.view(np.int16)).cuda() for h in layer] for layer in host]
    full = [torch.empty(total, dtype=torch.int16, device="cuda") for _ in range(2)]
    seen = torch.zeros(layers, total, dtype=torch.int16, device="cuda")
    main_s = torch.cuda.current_stream()
    side = torch.cuda.Stream()

    def gather(li, slot, stream):
        za.zero3_unit_gather_rows(shapes, world, shards[li], full[slot], stream=stream)

    def compute(li, slot):
        # a slow-ish stand-in, then record what the layer saw
        for _ in range(3):
            torch.mm(torch.ones(256, 256, device="cuda"), torch.ones(256, 256, device="cuda"))
        seen[li].copy_(full[slot])

    bench.prefetch_pass(layers, gather, compute, main_s, side)
    torch.cuda.synchronize()
    got = seen.cpu().numpy().view(np.uint16)
    for li in range(layers):
        assert (got[li] == oracle.unit_gather_rows(shapes, world, host[li])).all(), li
