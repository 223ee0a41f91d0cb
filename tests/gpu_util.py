"""Shared helpers of the GPU parity tests (CUDA path vs the oracle).

Inputs come from the seeded generator in synth/: the device generator fills
the GPU buffers, and the oracle gets the same bytes, either from the host
generator (windows) or as a host copy of the generator's device output whose
bytes are spot-checked against the host generator (whole-vector cases).
Nothing the oracle sees is computed by the library under test.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

# Tolerances of the parity bar: fp32 master/m/v within relative error 1e-6
# (exact where the oracle's value is 0); bf16 parameters within 1 ulp.
FP32_REL = 1e-6
BF16_ULP = 1


def ordered(bits: np.ndarray, width: int) -> np.ndarray:
    """Map float bit patterns to integers whose difference is the ulp distance."""
    b = bits.astype(np.int64)
    sign = 1 << (width - 1)
    return np.where(b & sign, -(b & (sign - 1)), b)


def ulp_distance_f32(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.abs(ordered(a.view(np.uint32), 32) - ordered(b.view(np.uint32), 32))


def ulp_distance_bf16(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.abs(ordered(a.astype(np.uint16), 16) - ordered(b.astype(np.uint16), 16))


def assert_f32_close(gpu: np.ndarray, ora: np.ndarray, what: str, exact: bool = True) -> None:
    """The bar: |gpu - ora| <= 1e-6 |ora|, equal where ora == 0, NaN where NaN.
    With exact=True also bit-for-bit equality (the kernel evaluates the oracle's
    operations in the oracle's order, so it is expected)."""
    assert gpu.shape == ora.shape, what
    nan = np.isnan(ora)
    assert (np.isnan(gpu) == nan).all(), f"{what}: NaN pattern differs"
    g, o = gpu[~nan].astype(np.float64), ora[~nan].astype(np.float64)
    with np.errstate(invalid="ignore"):  # inf - inf of equal infinities is fine
        bad = np.abs(g - o) > FP32_REL * np.abs(o)
    bad |= np.isinf(o) & (g != o)
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} elements off by > 1e-6 relative; "
                             f"first at {i}: gpu {g[i]!r} oracle {o[i]!r}")
    if exact:
        same = gpu[~nan].view(np.uint32) == ora[~nan].view(np.uint32)
        if not same.all():
            d = ulp_distance_f32(gpu[~nan], ora[~nan])
            raise AssertionError(f"{what}: {int((~same).sum())} elements not bit-exact "
                                 f"(max ulp distance {d.max()})")


def assert_bf16_close(gpu: np.ndarray, ora: np.ndarray, what: str, exact: bool = True) -> None:
    assert gpu.shape == ora.shape, what
    gf, of = oracle.bf16_to_f32(gpu), oracle.bf16_to_f32(ora)
    nan = np.isnan(of)
    assert (np.isnan(gf) == nan).all(), f"{what}: NaN pattern differs"
    d = ulp_distance_bf16(gpu[~nan], ora[~nan])
    assert d.max(initial=0) <= BF16_ULP, f"{what}: max bf16 ulp distance {d.max()}"
    if exact:
        same = gpu[~nan] == ora[~nan]
        assert same.all(), f"{what}: {int((~same).sum())} bf16 values not bit-exact"


def dev_fill(spec: synth.Spec, offset: int, n: int, kind: int, dtype, device="cuda") -> torch.Tensor:
    t = torch.empty(n, dtype=dtype, device=device)
    if n:
        synth.fill_dev(spec, offset, n, kind, t.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return t


def dev_fill_into(t: torch.Tensor, spec: synth.Spec, offset: int, kind: int) -> None:
    if t.numel():
        synth.fill_dev(spec, offset, t.numel(), kind, t.data_ptr(),
                       torch.cuda.current_stream().cuda_stream)


def to_host_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def to_host_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def spot_check_generated(t_host: np.ndarray, spec: synth.Spec, offset: int, kind: int,
                         samples: int = 4096, seed: int = 0) -> None:
    """The device generator's bytes equal the host generator's at random positions."""
    n = t_host.size
    if n == 0:
        return
    rng = np.random.default_rng(seed)
    pos = np.unique(np.concatenate([rng.integers(0, n, size=min(samples, n)), [0, n - 1]]))
    for p in pos[:: max(1, len(pos) // 64)]:
        ref = synth.fill_host(spec, offset + int(p), 1, kind)
        assert ref[0] == t_host[p], f"generator mismatch at {offset + p}"
    # one contiguous run too
    k = min(1024, n)
    ref = synth.fill_host(spec, offset, k, kind)
    assert (ref == t_host[:k]).all()


def bf16_tensor_bits(x: torch.Tensor) -> torch.Tensor:
    return x.view(torch.int16)


def oracle_step_parallel(numel, world, rank, grads, master, m, v, param, lr, b1, b2, eps, t, *,
                         i0=0, i1=None, grad_base=0, state_base=0, param_base=0,
                         threads=16, chunk=1 << 20) -> None:
    """oracle.zero_step over [i0, i1) split into disjoint windows run on a thread pool.

    The step is elementwise, so disjoint windows of the same arrays are
    independent; ctypes releases the GIL while the oracle's C loop runs."""
    from concurrent.futures import ThreadPoolExecutor

    if i1 is None:
        i1 = -(-numel // world) * world
    bounds = list(range(i0, i1, chunk)) + [i1]

    def run(k):
        oracle.zero_step(numel, world, rank, grads, master, m, v, param, lr, b1, b2, eps, t,
                         i0=bounds[k], i1=bounds[k + 1], grad_base=grad_base,
                         state_base=state_base, param_base=param_base)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(run, range(len(bounds) - 1)))
