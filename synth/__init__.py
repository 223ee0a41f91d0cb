"""Seeded synthetic inputs for the ZeRO Adam step (test and benchmark infrastructure).

Both the oracle side and the CUDA side take their inputs from here: the host
generator (``synth_host.c``, gcc) fills numpy arrays, the device generator
(``synth_dev.cu``, nvcc) fills device buffers, and the two are bit-identical
(``synth_core.h``).  The module holds none of the optimizer's arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_SO = os.path.join(_HERE, "libsynth_host.so")
_DEV_SO = os.path.join(_HERE, "libsynth_dev.so")
_HOST_SRC = [os.path.join(_HERE, "synth_host.c"), os.path.join(_HERE, "synth_core.h")]
_DEV_SRC = [os.path.join(_HERE, "synth_dev.cu"), os.path.join(_HERE, "synth_core.h")]

NORMAL, STUDENT_T3, CONSTANT = 0, 1, 2
OUT_F32, OUT_BF16 = 0, 1


class _Spec(ctypes.Structure):
    _fields_ = [
        ("seed", ctypes.c_uint64),
        ("stream", ctypes.c_uint32),
        ("rank", ctypes.c_uint32),
        ("step", ctypes.c_uint32),
        ("dist", ctypes.c_uint32),
        ("sigma", ctypes.c_float),
        ("outlier_value", ctypes.c_float),
        ("zero_thr", ctypes.c_uint64),
        ("outlier_thr", ctypes.c_uint64),
    ]


def _thr(p: float) -> int:
    """Probability p as a threshold on a uniform 64-bit word."""
    if p <= 0.0:
        return 0
    return min(int(p * 2.0**64), 2**64 - 1)


@dataclass(frozen=True)
class Spec:
    """Recipe of one synthetic buffer (see synth_core.h)."""

    seed: int
    stream: int
    rank: int = 0
    step: int = 0
    dist: int = NORMAL
    sigma: float = 1.0
    zero_frac: float = 0.0
    outlier_rate: float = 0.0
    outlier_value: float = 0.0

    def c(self) -> _Spec:
        return _Spec(self.seed, self.stream, self.rank, self.step, self.dist, self.sigma,
                     self.outlier_value, _thr(self.zero_frac), _thr(self.outlier_rate))


def _stale(so: str, srcs: list[str]) -> bool:
    if not os.path.exists(so):
        return True
    t = os.path.getmtime(so)
    return any(os.path.getmtime(s) > t for s in srcs)


def build_host(force: bool = False) -> str:
    if force or _stale(_HOST_SO, _HOST_SRC):
        tmp = _HOST_SO + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-fPIC", "-shared", "-o", tmp, _HOST_SRC[0], "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _HOST_SO)
    return _HOST_SO


def build_dev(force: bool = False, arch: str = "sm_103a") -> str:
    if force or _stale(_DEV_SO, _DEV_SRC):
        tmp = _DEV_SO + f".{os.getpid()}.tmp"
        nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
        comp = arch.replace("sm_", "compute_")
        cmd = [nvcc, "-O3", f"-gencode=arch={comp},code={arch}", "-std=c++17",
               "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off", "-shared",
               "-cudart", "shared", "-Xlinker",
               f"-rpath,{os.path.join(os.environ.get('CUDA_HOME', '/usr/local/cuda'), 'lib64')}",
               "-o", tmp, _DEV_SRC[0]]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _DEV_SO)
    return _DEV_SO


_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        lib = ctypes.CDLL(build_host())
        lib.synth_fill_host.argtypes = [ctypes.POINTER(_Spec), ctypes.c_int64, ctypes.c_int64,
                                        ctypes.c_void_p, ctypes.c_int]
        lib.synth_fill_host.restype = ctypes.c_int
        lib.synth_ln_host.argtypes = [ctypes.c_float]
        lib.synth_ln_host.restype = ctypes.c_float
        lib.synth_mix64_host.argtypes = [ctypes.c_uint64]
        lib.synth_mix64_host.restype = ctypes.c_uint64
        _host = lib
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        lib = ctypes.CDLL(build_dev())
        lib.synth_fill_dev.argtypes = [ctypes.POINTER(_Spec), ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
        lib.synth_fill_dev.restype = ctypes.c_int
        _dev = lib
    return _dev


def fill_host(spec: Spec, offset: int, n: int, kind: int) -> np.ndarray:
    """Elements [offset, offset+n) of the buffer, as float32 or uint16 (bf16 bits)."""
    out = np.empty(n, dtype=np.float32 if kind == OUT_F32 else np.uint16)
    cs = spec.c()
    rc = _host_lib().synth_fill_host(ctypes.byref(cs), offset, n,
                                     out.ctypes.data_as(ctypes.c_void_p), kind)
    if rc != 0:
        raise ValueError(f"synth_fill_host failed ({rc})")
    return out


def fill_dev(spec: Spec, offset: int, n: int, kind: int, ptr: int, stream: int = 0) -> None:
    """Device counterpart of fill_host, writing n elements at device address ptr."""
    cs = spec.c()
    rc = _dev_lib().synth_fill_dev(ctypes.byref(cs), offset, n, ctypes.c_void_p(ptr), kind,
                                   ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError(f"synth_fill_dev failed ({rc})")


def ln_host(s: float) -> float:
    return float(_host_lib().synth_ln_host(s))


def mix64_host(z: int) -> int:
    return int(_host_lib().synth_mix64_host(z))


if __name__ == "__main__":  # pragma: no cover - manual build entry
    build_host(force=True)
    if len(sys.argv) > 1 and sys.argv[1] == "dev":
        build_dev(force=True)
