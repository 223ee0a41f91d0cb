"""The oracle: a plain CPU statement of the ZeRO-1/2 Adam step (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and the
two share no code: the oracle is ``zero_oracle.c`` (plain C, gcc,
``-ffp-contract=off``), wrapped here with ctypes over numpy arrays.

Every function follows "ZeRO and FSDP: partitioning the optimizer states, the
gradients and the parameters" (AI infra handbooks): the planner follows the
"The three stages" table and ZeroAdam.__init__/_flatten; the step follows
ZeroAdam.step; the unit gather follows "ZeRO-3 and FSDP".  Pins: see
tests/test_oracle_pins.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libzero_oracle.so")
_SRC = [os.path.join(_HERE, "zero_oracle.c"), os.path.join(_HERE, "zero_oracle.h")]

MAX_WORLD = 1024


class _Plan(ctypes.Structure):
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


class _Scalars(ctypes.Structure):
    _fields_ = [(n, ctypes.c_float) for n in
                ("b1", "omb1", "b2", "omb2", "bc1", "bc2", "lr", "eps", "world")]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain IEEE binary32: no contraction, no fast-math).

    ZERO_ORACLE_SO names a prebuilt library to load instead; the oracle's own
    mutation test uses it to run the pins against deliberately broken copies.
    """
    override = os.environ.get("ZERO_ORACLE_SO")
    if override:
        return override
    stale = not os.path.exists(_SO) or any(os.path.getmtime(s) > os.path.getmtime(_SO)
                                           for s in _SRC)
    if force or stale:
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                        "-fPIC", "-shared", "-o", tmp, _SRC[0], "-lm"], check=True)
        os.replace(tmp, _SO)
    return _SO


_lib = None


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.POINTER
        lib.oracle_plan.argtypes = [ctypes.c_int64, ctypes.c_int32, P(_Plan)]
        lib.oracle_plan.restype = ctypes.c_int
        lib.oracle_f32_to_bf16_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
        lib.oracle_f32_to_bf16_array.restype = None
        lib.oracle_scalars.argtypes = [ctypes.c_double] * 4 + [ctypes.c_int64, ctypes.c_int32,
                                                               P(_Scalars)]
        lib.oracle_scalars.restype = None
        lib.oracle_zero_step.argtypes = (
            [P(_Plan), ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
             ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
             ctypes.c_void_p, ctypes.c_int64] + [ctypes.c_double] * 4 + [ctypes.c_int64])
        lib.oracle_zero_step.restype = ctypes.c_int
        lib.oracle_zero_step_ex.argtypes = (
            [P(_Plan), ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
             ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
             ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64]
            + [ctypes.c_double] * 4 + [ctypes.c_int64])
        lib.oracle_zero_step_ex.restype = ctypes.c_int
        lib.oracle_dp_step.argtypes = (
            [ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
             ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_double] * 4 + [ctypes.c_int64])
        lib.oracle_dp_step.restype = ctypes.c_int
        lib.oracle_unit_gather.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p,
                                           ctypes.c_void_p]
        lib.oracle_unit_gather.restype = ctypes.c_int
        lib.oracle_unit_gather_rows.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_unit_gather_rows.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> ctypes.c_void_p:
    return a.ctypes.data_as(ctypes.c_void_p)


def _ptr_array(arrs, dtype=np.uint16) -> ctypes.Array:
    for a in arrs:
        assert a.dtype == dtype and a.flags.c_contiguous
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


def plan(numel: int, world: int) -> dict:
    """Shard/pad layout and per-card model-state bytes (see oracle_plan)."""
    p = _Plan()
    if _L().oracle_plan(numel, world, ctypes.byref(p)) != 0:
        raise ValueError(f"invalid plan ({numel}, {world})")
    return {name: getattr(p, name) for name, _ in _Plan._fields_}


def _plan_struct(numel: int, world: int) -> _Plan:
    p = _Plan()
    if _L().oracle_plan(numel, world, ctypes.byref(p)) != 0:
        raise ValueError(f"invalid plan ({numel}, {world})")
    return p


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even binary32 -> bf16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _L().oracle_f32_to_bf16_array(_ptr(x), _ptr(out), x.size)
    return out


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 bits -> binary32 (exact)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def scalars(lr, beta1, beta2, eps, t, world) -> dict:
    s = _Scalars()
    _L().oracle_scalars(lr, beta1, beta2, eps, t, world, ctypes.byref(s))
    return {name: getattr(s, name) for name, _ in _Scalars._fields_}


def zero_step(numel, world, rank, grads, master, m, v, param, lr, beta1, beta2, eps, t, *,
              i0=0, i1=None, grad_base=0, state_base=0, param_base=0, grad_f32=False,
              acc_bf16=False) -> None:
    """ZeroAdam.step for one rank (rank >= 0) or all ranks (rank = -1), in place.

    Arrays are addressed by global flat index minus their base (see
    oracle_zero_step); only global indices in [i0, i1) are touched.  grads are
    uint16 (bf16 bits), or float32 with grad_f32; acc_bf16 selects the
    bf16-rounded running sum (a variant, not the method).
    """
    p = _plan_struct(numel, world)
    if i1 is None:
        i1 = p.padded
    assert len(grads) == world
    for a in (master, m, v):
        assert a.dtype == np.float32 and a.flags.c_contiguous
    assert param.dtype == np.uint16 and param.flags.c_contiguous
    ptrs = _ptr_array(grads, np.float32 if grad_f32 else np.uint16)
    if not grad_f32 and not acc_bf16:
        rc = _L().oracle_zero_step(ctypes.byref(p), rank, i0, i1, ptrs, grad_base, _ptr(master),
                                   _ptr(m), _ptr(v), state_base, _ptr(param), param_base,
                                   lr, beta1, beta2, eps, t)
    else:
        rc = _L().oracle_zero_step_ex(ctypes.byref(p), rank, i0, i1, ptrs, grad_base,
                                      int(grad_f32), int(acc_bf16), _ptr(master), _ptr(m),
                                      _ptr(v), state_base, _ptr(param), param_base,
                                      lr, beta1, beta2, eps, t)
    if rc != 0:
        raise ValueError(f"oracle_zero_step failed ({rc})")


def dp_step(numel, world, grads, master, m, v, param, lr, beta1, beta2, eps, t) -> None:
    """Unpartitioned data-parallel Adam on the rank-averaged gradient, in place."""
    ptrs = _ptr_array(grads)
    rc = _L().oracle_dp_step(numel, world, ptrs, _ptr(master), _ptr(m), _ptr(v), _ptr(param),
                             lr, beta1, beta2, eps, t)
    if rc != 0:
        raise ValueError(f"oracle_dp_step failed ({rc})")


def unit_gather(unit_numel: int, world: int, shards) -> np.ndarray:
    """ZeRO-3 unit all-gather: N bf16 shards of ceil(U/N) -> the unit's U elements."""
    full = np.zeros(unit_numel, dtype=np.uint16)
    rc = _L().oracle_unit_gather(unit_numel, world, _ptr_array(shards), _ptr(full))
    if rc != 0:
        raise ValueError("oracle_unit_gather failed")
    return full


def rows_layout(shapes, world):
    """Sizes of the FSDP2-style row-sharded layout: (shard elements per rank, unit elements)."""
    shard = sum(-(-r // world) * c for r, c in shapes)
    return shard, sum(r * c for r, c in shapes)


def unit_gather_rows(shapes, world: int, shards) -> np.ndarray:
    """FSDP2-style unit gather: tensors (rows, cols) sharded by rows -> the full unit."""
    rows = np.array([r for r, _ in shapes], np.int64)
    cols = np.array([c for _, c in shapes], np.int64)
    shard_len, total = rows_layout(shapes, world)
    for s in shards:
        assert s.size == shard_len
    full = np.zeros(total, dtype=np.uint16)
    rc = _L().oracle_unit_gather_rows(len(shapes), _ptr(rows), _ptr(cols), world,
                                      _ptr_array(shards), _ptr(full))
    if rc != 0:
        raise ValueError("oracle_unit_gather_rows failed")
    return full
