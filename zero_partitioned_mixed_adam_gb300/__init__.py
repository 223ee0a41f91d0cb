"""ZeRO stage-1/2 mixed-precision Adam step on one GB300: Python binding.

A thin ctypes layer over libzeroadam.so (include/zeroadam.h).  It marshals
arguments only: every step of the optimizer runs in the library's CUDA
kernels.  PyTorch provides device memory and streams.  There is no CPU
fallback: importing this package fails loudly when the library is missing.

The method: "ZeRO and FSDP: partitioning the optimizer states, the gradients
and the parameters" (AI infra handbooks), "Implementing ZeRO's Adam from
scratch" (ZeroAdam) and "ZeRO-3 and FSDP" (unit all-gather).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libzeroadam.so")

ZERO_OK = 0
ZERO_ALL_RANKS = -1
ZERO_GRAD_FULL, ZERO_GRAD_SHARD, ZERO_GRAD_WINDOW = 0, 1, 2
ZERO_GRAD_LAYOUT_MASK = 0x0F
ZERO_GRAD_F32, ZERO_ACC_BF16 = 0x10, 0x20
ZERO_PARAM_FULL, ZERO_PARAM_SHARD = 0, 1
ZERO_MAX_WORLD = 1024
ZERO_MAX_UNIT_TENSORS = 256

ERRORS = {
    -1: "ZERO_E_NULLPTR", -2: "ZERO_E_WORLD", -3: "ZERO_E_NUMEL", -4: "ZERO_E_RANK",
    -5: "ZERO_E_STEP", -6: "ZERO_E_ALIGN", -7: "ZERO_E_HPARAM", -8: "ZERO_E_LAYOUT",
    -9: "ZERO_E_PLAN", -10: "ZERO_E_ALIAS", -11: "ZERO_E_LAUNCH", -12: "ZERO_E_DEVICE",
    -13: "ZERO_E_RANGE", -14: "ZERO_E_SHAPE", -15: "ZERO_E_TIMEOUT", -16: "ZERO_E_HOOK",
}

# Every symbol include/zeroadam.h declares.
EXPORTS = ("zero_plan", "zero_adam_step", "zero_adam_step_range", "zero3_unit_gather",
           "zero3_unit_gather_rows", "zero3_unit_step", "zero_device_status",
           "zero_test_withhold_copies", "zero_strerror", "zero_version")


class ZeroError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        self.code = ERRORS.get(status, str(status))
        super().__init__(f"{what}: {self.code}: {strerror(status)}")


class ZeroPlan(ctypes.Structure):
    """zero_plan_t: shard layout and per-card model-state/communication bytes."""

    _fields_ = [
        ("numel", ctypes.c_int64), ("world", ctypes.c_int64), ("shard", ctypes.c_int64),
        ("pad", ctypes.c_int64), ("padded", ctypes.c_int64),
        ("bytes_dp", ctypes.c_uint64), ("bytes_z1", ctypes.c_uint64),
        ("bytes_z2", ctypes.c_uint64), ("bytes_z3", ctypes.c_uint64),
        ("formula_dp", ctypes.c_double), ("formula_z1", ctypes.c_double),
        ("formula_z2", ctypes.c_double), ("formula_z3", ctypes.c_double),
        ("state_bytes_rank", ctypes.c_uint64),
        ("comm_dp", ctypes.c_double), ("comm_z1", ctypes.c_double),
        ("comm_z2", ctypes.c_double), ("comm_z3", ctypes.c_double),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; "
            "g.build()' or python zero_partitioned_mixed_adam_gb300/build.py)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.zero_plan.argtypes = [i64, i32, ctypes.POINTER(ZeroPlan)]
    lib.zero_plan.restype = ctypes.c_int
    lib.zero_adam_step.argtypes = [ctypes.POINTER(ZeroPlan), i32, vp, i32, vp, vp, vp, vp, i32,
                                   dbl, dbl, dbl, dbl, i64, vp]
    lib.zero_adam_step.restype = ctypes.c_int
    lib.zero_adam_step_range.argtypes = [ctypes.POINTER(ZeroPlan), i32, i64, i64, vp, i32, vp, vp,
                                         vp, vp, i32, dbl, dbl, dbl, dbl, i64, vp]
    lib.zero_adam_step_range.restype = ctypes.c_int
    lib.zero3_unit_gather.argtypes = [ctypes.POINTER(ZeroPlan), vp, vp, vp]
    lib.zero3_unit_gather.restype = ctypes.c_int
    lib.zero3_unit_step.argtypes = [ctypes.POINTER(ZeroPlan), i32, vp, vp, vp, i32, vp, vp, vp,
                                    vp, i32, dbl, dbl, dbl, dbl, i64, vp]
    lib.zero3_unit_step.restype = ctypes.c_int
    lib.zero3_unit_gather_rows.argtypes = [i32, vp, vp, i32, vp, vp, vp]
    lib.zero3_unit_gather_rows.restype = ctypes.c_int
    lib.zero_device_status.argtypes = []
    lib.zero_device_status.restype = ctypes.c_int
    lib.zero_test_withhold_copies.argtypes = [ctypes.c_int]
    lib.zero_test_withhold_copies.restype = ctypes.c_int
    lib.zero_strerror.argtypes = [ctypes.c_int]
    lib.zero_strerror.restype = ctypes.c_char_p
    lib.zero_version.argtypes = []
    lib.zero_version.restype = ctypes.c_int
    return lib


_lib = _load()


def strerror(status: int) -> str:
    return _lib.zero_strerror(status).decode()


def _addr(x) -> int:
    """Device address of a tensor (data_ptr) or a raw integer address."""
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


class PointerArray:
    """The device addresses of a fixed list of buffers, marshalled once.

    Pass it wherever a call takes a sequence of buffers (gradients, shards): a
    training loop hands the same buffers to every step, and building the C
    array of N addresses is most of a call's host time at large N.  It keeps
    references to the buffers, so they stay alive as long as the array does;
    it records each buffer's address when built and does not follow a buffer
    whose storage is replaced afterwards (build a new array then)."""

    __slots__ = ("arr", "buffers")

    def __init__(self, buffers):
        self.buffers = tuple(buffers)
        self.arr = (ctypes.c_void_p * len(self.buffers))(*[_addr(b) for b in self.buffers])

    def __len__(self) -> int:
        return len(self.buffers)


def pointer_array(buffers) -> PointerArray:
    """A reusable PointerArray of `buffers` (tensors or raw addresses)."""
    return PointerArray(buffers)


def _ptrs(buffers):
    """The C array of addresses: a PointerArray's own, else built from the sequence."""
    if isinstance(buffers, PointerArray):
        return buffers.arr
    return (ctypes.c_void_p * len(buffers))(*[_addr(b) for b in buffers])


def _stream_handle(stream) -> int:
    if stream is None:
        try:
            import torch
            return int(torch.cuda.current_stream().cuda_stream)
        except Exception:
            return 0
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def zero_plan(numel: int, world: int) -> ZeroPlan:
    p = ZeroPlan()
    rc = _lib.zero_plan(numel, world, ctypes.byref(p))
    if rc != ZERO_OK:
        raise ZeroError(rc, "zero_plan")
    return p


def zero_adam_step(plan: ZeroPlan, rank: int, grads, master, m, v, param, *, lr: float,
                   beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8, t: int,
                   grad_layout: int = ZERO_GRAD_FULL, param_layout: int = ZERO_PARAM_FULL,
                   stream=None) -> None:
    """One fused ZeRO Adam step (reduce-scatter + Adam + bf16 all-gather) on the GPU.

    grads: sequence of `world` bf16 device buffers (tensors or addresses), or a
    PointerArray of them (pointer_array: marshalled once, reused every step);
    master/m/v: fp32 device buffers; param: bf16 device buffer.  Layouts and
    index conventions are those of zero_adam_step in include/zeroadam.h.
    """
    if len(grads) != plan.world:
        raise ValueError(f"expected {plan.world} gradient buffers, got {len(grads)}")
    ptrs = _ptrs(grads)
    rc = _lib.zero_adam_step(ctypes.byref(plan), rank, ptrs, grad_layout, _addr(master),
                             _addr(m), _addr(v), _addr(param), param_layout, lr, beta1, beta2,
                             eps, t, _stream_handle(stream))
    if rc != ZERO_OK:
        raise ZeroError(rc, "zero_adam_step")


def zero_adam_step_range(plan: ZeroPlan, rank: int, begin: int, end: int, grads, master, m, v,
                         param, *, lr: float, beta1: float = 0.9, beta2: float = 0.999,
                         eps: float = 1e-8, t: int, grad_layout: int = ZERO_GRAD_WINDOW,
                         param_layout: int = ZERO_PARAM_FULL, stream=None) -> None:
    """The step on the global flat window [begin, end) only (one ZeRO-2 bucket).

    With ZERO_GRAD_WINDOW (the default here) each gradient buffer holds only the
    window: element i at grads[k][i - begin].
    """
    if len(grads) != plan.world:
        raise ValueError(f"expected {plan.world} gradient buffers, got {len(grads)}")
    ptrs = _ptrs(grads)
    rc = _lib.zero_adam_step_range(ctypes.byref(plan), rank, begin, end, ptrs, grad_layout,
                                   _addr(master), _addr(m), _addr(v), _addr(param), param_layout,
                                   lr, beta1, beta2, eps, t, _stream_handle(stream))
    if rc != ZERO_OK:
        raise ZeroError(rc, "zero_adam_step_range")


def zero3_unit_gather(unit_plan: ZeroPlan, shards, full, stream=None) -> None:
    """ZeRO-3 unit all-gather: the `world` bf16 shards -> the unit's full bf16 buffer."""
    if len(shards) != unit_plan.world:
        raise ValueError(f"expected {unit_plan.world} shards, got {len(shards)}")
    ptrs = _ptrs(shards)
    rc = _lib.zero3_unit_gather(ctypes.byref(unit_plan), ptrs, _addr(full),
                                _stream_handle(stream))
    if rc != ZERO_OK:
        raise ZeroError(rc, "zero3_unit_gather")


def zero3_unit_step(unit_plan: ZeroPlan, rank: int, shards, full, grads, master, m, v, param, *,
                    lr: float, beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8,
                    t: int, grad_layout: int = ZERO_GRAD_SHARD,
                    param_layout: int = ZERO_PARAM_SHARD, stream=None) -> None:
    """One ZeRO-3 unit: the gather of the `world` bf16 shards into `full` and rank
    `rank`'s fused step, in one launch (the same results as zero3_unit_gather followed
    by zero_adam_step; the two parts' buffers must be disjoint)."""
    if len(shards) != unit_plan.world or len(grads) != unit_plan.world:
        raise ValueError(f"expected {unit_plan.world} shards and gradient buffers")
    sp, gp = _ptrs(shards), _ptrs(grads)
    rc = _lib.zero3_unit_step(ctypes.byref(unit_plan), rank, sp, _addr(full), gp, grad_layout,
                              _addr(master), _addr(m), _addr(v), _addr(param), param_layout, lr,
                              beta1, beta2, eps, t, _stream_handle(stream))
    if rc != ZERO_OK:
        raise ZeroError(rc, "zero3_unit_step")


def rows_layout(shapes, world: int):
    """(elements of one rank's shard, elements of the unit) of the FSDP2-style layout."""
    return (sum(-(-r // world) * c for r, c in shapes), sum(r * c for r, c in shapes))


def zero3_unit_gather_rows(shapes, world: int, shards, full, stream=None) -> None:
    """FSDP2-style gather: tensors of shapes [(rows, cols), ...] sharded by rows across
    `world` ranks (rank r holds rows [r*R, (r+1)*R), R = ceil(rows/world), of each
    tensor, back to back) -> the unit's tensors back to back."""
    if len(shards) != world:
        raise ValueError(f"expected {world} shards, got {len(shards)}")
    n = len(shapes)
    rows = (ctypes.c_int64 * max(n, 1))(*[int(r) for r, _ in shapes])
    cols = (ctypes.c_int64 * max(n, 1))(*[int(c) for _, c in shapes])
    ptrs = _ptrs(shards)
    rc = _lib.zero3_unit_gather_rows(n, rows, cols, world, ptrs, _addr(full),
                                     _stream_handle(stream))
    if rc != ZERO_OK:
        raise ZeroError(rc, "zero3_unit_gather_rows")


def device_status() -> int:
    """ZERO_OK, or ZERO_E_TIMEOUT if a kernel gave up a bounded wait since the last call
    (synchronises the current device, then reads and clears the words)."""
    return _lib.zero_device_status()


def check_device(what: str = "device_status") -> None:
    """Raise ZeroError unless every bounded wait since the last check completed."""
    rc = _lib.zero_device_status()
    if rc != ZERO_OK:
        raise ZeroError(rc, what)


def test_withhold_copies(on: bool) -> bool:
    """Test hook: while on, the TMA-staged kernels issue no copies, so their bounded
    waits run out (zero_device_status then reports ZERO_E_TIMEOUT).  Needs
    ZEROADAM_TEST_HOOKS=1 in the environment.  Returns the previous setting."""
    rc = _lib.zero_test_withhold_copies(1 if on else 0)
    if rc < 0:
        raise ZeroError(rc, "zero_test_withhold_copies")
    return bool(rc)


def version() -> int:
    return _lib.zero_version()


def raw_lib() -> ctypes.CDLL:
    """The loaded libzeroadam.so (for callers that pass their own pointers)."""
    return _lib


__all__ = ["zero_plan", "zero_adam_step", "zero_adam_step_range", "zero3_unit_gather",
           "zero3_unit_gather_rows", "pointer_array", "PointerArray", "zero3_unit_step", "rows_layout", "device_status",
           "check_device", "test_withhold_copies",
           "ZeroPlan", "ZeroError", "strerror", "version", "raw_lib", "ZERO_ALL_RANKS",
           "ZERO_GRAD_FULL", "ZERO_GRAD_SHARD", "ZERO_GRAD_WINDOW", "ZERO_GRAD_F32",
           "ZERO_ACC_BF16", "ZERO_PARAM_FULL", "ZERO_PARAM_SHARD", "ZERO_MAX_WORLD",
           "ZERO_MAX_UNIT_TENSORS", "EXPORTS", "LIB_PATH"]
