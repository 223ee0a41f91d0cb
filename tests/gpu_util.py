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


# ------------------------------------------------- full-size parity on sampled windows

CHUNK = 1 << 24   # random chunks compared element by element
EDGE = 1 << 20    # elements compared at the start and the end of every rank's range
HALO = 16         # elements compared on each side of every shard or unit boundary


def sample_windows(lo, hi, rank_ranges, rng, n_chunks=3, chunk=CHUNK, edge=EDGE, halo=HALO,
                   boundaries=()):
    """Global index windows [a, b) inside [lo, hi) that a full-size parity test compares:
    every element of `n_chunks` random `chunk`-element chunks, the first and last `edge`
    elements of each rank range, and every index within `halo` of a boundary (each rank
    range's ends and `boundaries`).  Overlapping or touching windows are merged."""
    ws = []
    for a, b in rank_ranges:
        a, b = max(lo, a), min(hi, b)
        if b > a:
            ws += [(a, min(b, a + edge)), (max(a, b - edge), b)]
    for x in [a for a, _ in rank_ranges] + [b for _, b in rank_ranges] + list(boundaries):
        ws.append((max(lo, x - halo), min(hi, x + halo)))
    for _ in range(n_chunks):
        a = int(rng.integers(lo, max(lo + 1, hi - chunk + 1)))
        ws.append((a, min(hi, a + chunk)))
    ws = sorted((a, b) for a, b in ws if b > a)
    merged = []
    for a, b in ws:
        if merged and a <= merged[-1][1]:
            merged[-1] = (merged[-1][0], max(merged[-1][1], b))
        else:
            merged.append((a, b))
    return merged


def window_elements(windows):
    return sum(b - a for a, b in windows)


class WindowOracle:
    """The oracle's state on a set of global index windows of one workload, stepped
    with the same gradient bytes the device saw.  Initial master weights come from the
    host generator; moments start at zero."""

    def __init__(self, numel, world, rank, windows, master_spec, hparams):
        self.numel, self.world, self.rank = numel, world, rank
        self.windows = windows
        self.hp = hparams
        self.w = [synth.fill_host(master_spec, a, b - a, synth.OUT_F32) for a, b in windows]
        self.m = [np.zeros(b - a, np.float32) for a, b in windows]
        self.v = [np.zeros(b - a, np.float32) for a, b in windows]
        self.p = [np.zeros(b - a, np.uint16) for a, b in windows]

    def step(self, t, grads, threads=16, sub=1 << 20):
        """grads[j][k]: rank k's bf16 gradient on window j (uint16, the window's length)."""
        from concurrent.futures import ThreadPoolExecutor
        lr, b1, b2, eps = self.hp
        jobs = []
        for j, (a, b) in enumerate(self.windows):
            for i0 in range(a, b, sub):
                jobs.append((j, i0, min(b, i0 + sub)))

        def run(job):
            j, i0, i1 = job
            a = self.windows[j][0]
            oracle.zero_step(self.numel, self.world, self.rank, grads[j], self.w[j], self.m[j],
                             self.v[j], self.p[j], lr, b1, b2, eps, t, i0=i0, i1=i1,
                             grad_base=a, state_base=a, param_base=a)

        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(run, jobs))

    def compare(self, master, m, v, param, state_first, param_first, what):
        """Device state (index = global - state_first) and bf16 parameters (index =
        global - param_first) against the oracle on every window."""
        for j, (a, b) in enumerate(self.windows):
            s = slice(a - state_first, b - state_first)
            ps = slice(a - param_first, b - param_first)
            tag = f"{what} [{a},{b})"
            assert_f32_close(to_host_f32(master[s]), self.w[j], f"{tag} master")
            assert_f32_close(to_host_f32(m[s]), self.m[j], f"{tag} m")
            assert_f32_close(to_host_f32(v[s]), self.v[j], f"{tag} v")
            assert_bf16_close(to_host_u16(param[ps]), self.p[j], f"{tag} param")


def device_grad_windows(grads, windows, first, specs=None, check_every=4, seed=0):
    """Host copies of the device gradient buffers on each window (buffer index = global -
    first): out[j][k].  With specs (rank k's generator recipe, indexed by global
    position), some windows' bytes are spot-checked against the host generator."""
    out = []
    for j, (a, b) in enumerate(windows):
        row = []
        for k, g in enumerate(grads):
            h = to_host_u16(g[a - first:b - first]).copy()
            if specs is not None and (j + k) % check_every == 0:
                spot_check_generated(h, specs[k], a, synth.OUT_BF16, samples=256,
                                     seed=seed + 31 * j + k)
            row.append(h)
        out.append(row)
    return out
