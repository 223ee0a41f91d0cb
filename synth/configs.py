"""The five synthetic workloads of the ZeRO Adam step: sizes and input recipes.

Sizes only and draw recipes: no optimizer arithmetic lives here.

  tiny      Psi = 1,000,003 = [1000x512] + [512] + [487,491] flattened; N = 4, all ranks,
            grads bf16 N(0,1e-3), master N(0,0.02), m = v = 0, 3 steps, seed 0.
  gpt2      GPT-2-small flat vector, Psi = 124,439,808, N = 8, all ranks, grads bf16
            N(0,1e-3) with a 10 % exact-zero mask shared by the ranks, 10 steps.
  1p3b      Psi = 1.3e9 (24 layers, d 2048, MLP 8192, the rest embeddings), N = 16, all ranks,
            grads bf16 Student-t(3) x 1e-3 with +-1e2 outliers at rate 1e-6, m and v from
            5 prior steps, timed from t = 6.
  7b_rank3  Psi = 7e9 (Llama-style 7B), N = 8, rank 3 only: 8 bf16 gradient slices of its
            875M-element shard, fp32 master/m/v of the shard, bf16 output into the full
            7e9-element parameter buffer.  7b_rank3_prewarm: the same with m and v from
            5 prior steps, timed from t = 6.
  unit      ZeRO-3 units of U in {2^20, 2^24, 202,383,360 (one Llama-7B layer), 2^29} elements,
            N in {2, 8, 64}: gather the N bf16 parameter shards, then rank 0's step on its
            shard from N bf16 gradient slices.
"""
from __future__ import annotations

from dataclasses import dataclass, field

from . import NORMAL, STUDENT_T3, Spec

# synth stream ids (one per kind of buffer)
STREAM_GRAD, STREAM_MASTER, STREAM_PARAM_SHARD = 1, 2, 3

GPT2_SMALL_SHAPES = (
    [(50257, 768), (1024, 768)]
    + [(768,), (768,), (768, 2304), (2304,), (768, 768), (768,), (768,), (768,),
       (768, 3072), (3072,), (3072, 768), (768,)] * 12
    + [(768,), (768,)]
)


def _numel(shapes) -> int:
    n = 0
    for s in shapes:
        k = 1
        for d in s:
            k *= d
        n += k
    return n


@dataclass(frozen=True)
class StepWorkload:
    name: str
    numel: int
    world: int
    rank: int = -1              # -1: every rank; else the one rank stepped
    grad_layout: str = "full"   # "full": rank k's whole padded gradient; "shard": its slice
    param_layout: str = "full"  # "full": the whole flat bf16 buffer; "shard": the rank's shard
    steps: int = 3
    prewarm: int = 0            # steps run before the first checked/timed one
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    seed: int = 0
    grad_dist: int = NORMAL
    grad_sigma: float = 1e-3
    grad_zero_frac: float = 0.0
    outlier_rate: float = 0.0
    outlier_value: float = 0.0
    master_sigma: float = 0.02
    shapes: tuple = field(default=())
    grad_f32: bool = False      # gradient buffers hold fp32 (the page's runnable demo)
    acc_bf16: bool = False      # the sum over ranks is rounded to bf16 after every addition

    @property
    def shard(self) -> int:
        return -(-self.numel // self.world)

    def grad_spec(self, k: int, step: int) -> Spec:
        """Rank k's gradient at step t (1-based), indexed by global flat position."""
        return Spec(seed=self.seed, stream=STREAM_GRAD, rank=k, step=step, dist=self.grad_dist,
                    sigma=self.grad_sigma, zero_frac=self.grad_zero_frac,
                    outlier_rate=self.outlier_rate, outlier_value=self.outlier_value)

    def master_spec(self) -> Spec:
        """Initial fp32 master weights, indexed by global flat position."""
        return Spec(seed=self.seed, stream=STREAM_MASTER, sigma=self.master_sigma)


TINY = StepWorkload("tiny", numel=_numel([(1000, 512), (512,), (487491,)]), world=4, steps=3,
                    shapes=((1000, 512), (512,), (487491,)))
GPT2 = StepWorkload("gpt2", numel=_numel(GPT2_SMALL_SHAPES), world=8, steps=10,
                    grad_zero_frac=0.1)
B1P3 = StepWorkload("1p3b", numel=1_300_000_000, world=16, steps=1, prewarm=5,
                    grad_dist=STUDENT_T3, outlier_rate=1e-6, outlier_value=1e2)
B7_RANK3 = StepWorkload("7b_rank3", numel=7_000_000_000, world=8, rank=3, grad_layout="shard",
                        steps=1)
# the same rank with five steps of moment history before the first timed step
B7_RANK3_PREWARM = StepWorkload("7b_rank3_prewarm", numel=7_000_000_000, world=8, rank=3,
                                grad_layout="shard", steps=1, prewarm=5)

assert TINY.numel == 1_000_003 and TINY.shard == 250_001
assert GPT2.numel == 124_439_808 and GPT2.shard == 15_554_976
assert B1P3.shard == 81_250_000 and B7_RANK3.shard == 875_000_000

UNIT_SIZES = (1_048_576, 16_777_216, 202_383_360, 536_870_912)
UNIT_WORLDS = (2, 8, 64)
assert 4 * 4096 * 4096 + 3 * 4096 * 11008 + 2 * 4096 == UNIT_SIZES[2]


def unit_workload(unit_numel: int, world: int) -> StepWorkload:
    """One ZeRO-3 unit: rank 0's step on its shard from N gradient slices."""
    return StepWorkload(f"unit{unit_numel}_n{world}", numel=unit_numel, world=world, rank=0,
                        grad_layout="shard", param_layout="shard", steps=1)


def unit_shard_step_workload(unit_numel: int, world: int) -> StepWorkload:
    """The same unit's rank-0 step alone (no gather before it): the step measured on
    its own, with the same inputs as unit_workload's step."""
    return StepWorkload(f"shard{unit_numel}_n{world}", numel=unit_numel, world=world, rank=0,
                        grad_layout="shard", param_layout="shard", steps=1)


def unit_shard_spec(unit_numel: int, world: int, r: int) -> Spec:
    """Rank r's bf16 parameter shard of a ZeRO-3 unit (input of the gather)."""
    return Spec(seed=unit_numel % 1000003 + world, stream=STREAM_PARAM_SHARD, rank=r, sigma=0.02)


WORKLOADS = {w.name: w for w in (TINY, GPT2, B1P3, B7_RANK3, B7_RANK3_PREWARM)}
