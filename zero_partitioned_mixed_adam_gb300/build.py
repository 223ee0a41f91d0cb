"""Build libzeroadam.so in-tree for sm_103a (nvcc; no cmake, no torch extension).

Each translation unit compiles in parallel; the library links the shared CUDA
runtime, so it shares one runtime with PyTorch when both are loaded.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "libzeroadam.so")
OBJ_DIR = os.path.join(ROOT, "_build", "zeroadam")
SOURCES = ["capi.cpp", "adam_step.cu", "unit_gather.cu"]
HEADERS = ([os.path.join(CSRC, h) for h in sorted(os.listdir(CSRC)) if h.endswith(".h")]
           + [os.path.join(ROOT, "include", "zeroadam.h")])
ARCH = "sm_103a"


def _cuda_home() -> str:
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _flags(verbose_ptxas: bool) -> list[str]:
    comp = ARCH.replace("sm_", "compute_")
    f = ["-O3", "-std=c++17", f"-gencode=arch={comp},code={ARCH}", "-lineinfo",
         "-Xcompiler", "-fPIC", "-Xcompiler", "-O2", "-I", os.path.join(ROOT, "include")]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    nvcc = os.path.join(_cuda_home(), "bin", "nvcc")
    os.makedirs(OBJ_DIR, exist_ok=True)
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(OBJ_DIR, src + ".o")
        objs.append(o)
        if force or verbose_ptxas or _stale(o, [s] + HEADERS):
            jobs.append([nvcc, "-c", s, "-o", o] + _flags(verbose_ptxas))

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        logs = list(ex.map(run, jobs))
    if verbose_ptxas:
        for log in logs:
            sys.stdout.write(log)
    if force or jobs or _stale(OUT, objs):
        tmp = OUT + f".{os.getpid()}.tmp"
        run([nvcc, "-shared", "-cudart", "shared", "-o", tmp] + objs +
            [f"-gencode=arch={ARCH.replace('sm_', 'compute_')},code={ARCH}",
             "-Xlinker", f"-rpath,{os.path.join(_cuda_home(), 'lib64')}"])
        os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv)
    print(OUT)
