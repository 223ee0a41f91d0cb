"""Tracing: every entry point that launches or waits for GPU work opens an NVTX range
named after itself for the whole call, error returns included.  A small NVTX injection
library (tests/c/nvtx_trace.c) records the pushes and pops of a child process that calls
the entry points with arguments they reject before touching a GPU, so this runs on CPU."""
import os
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")

CHILD = textwrap.dedent("""
    import ctypes, sys
    sys.path.insert(0, {root!r})
    import zero_partitioned_mixed_adam_gb300 as za
    lib = za.raw_lib()
    codes = [
        lib.zero_adam_step(None, -1, None, 0, None, None, None, None, 0,
                           1e-3, 0.9, 0.999, 1e-8, 1, None),
        lib.zero_adam_step_range(None, -1, 0, 10, None, 0, None, None, None, None, 0,
                                 1e-3, 0.9, 0.999, 1e-8, 1, None),
        lib.zero3_unit_gather(None, None, None, None),
        lib.zero3_unit_gather_rows(0, None, None, 1, None, None, None),
        lib.zero_device_status(),   # ZERO_E_DEVICE without a GPU, ZERO_OK with one
        lib.zero3_unit_step(None, 0, None, None, None, 1, None, None, None, None, 1,
                            1e-3, 0.9, 0.999, 1e-8, 1, None),
    ]
    plan = za.ZeroPlan()
    codes.append(lib.zero_plan(1000, 4, ctypes.byref(plan)))   # host only: not traced
    tracer = ctypes.CDLL({so!r})
    tracer.nvtx_trace_log.restype = ctypes.c_char_p
    print(",".join(str(c) for c in codes))
    print(tracer.nvtx_trace_log().decode())
""")


@pytest.fixture(scope="module")
def tracer_so(tmp_path_factory):
    so = str(tmp_path_factory.mktemp("nvtx") / "libnvtx_trace.so")
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-O2", "-shared", "-fPIC",
                    "-I", os.path.join(CUDA, "include"),
                    os.path.join(ROOT, "tests", "c", "nvtx_trace.c"), "-o", so], check=True)
    return so


def test_entry_points_open_and_close_their_ranges(tracer_so):
    env = dict(os.environ, NVTX_INJECTION64_PATH=tracer_so)
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, so=tracer_so)],
                       capture_output=True, text=True, timeout=120, env=env)
    assert r.returncode == 0, r.stderr
    codes, log = r.stdout.strip().splitlines()
    import zero_partitioned_mixed_adam_gb300 as za
    e = {v: k for k, v in za.ERRORS.items()}
    c = codes.split(",")
    assert c[:4] == [str(e["ZERO_E_NULLPTR"]), str(e["ZERO_E_NULLPTR"]),
                     str(e["ZERO_E_NULLPTR"]), str(e["ZERO_E_SHAPE"])]
    assert c[4] in ("0", str(e["ZERO_E_DEVICE"])) and c[5] == str(e["ZERO_E_NULLPTR"])
    assert c[6] == "0"
    assert log == ("+zero_adam_step;-;+zero_adam_step_range;-;+zero3_unit_gather;-;"
                   "+zero3_unit_gather_rows;-;+zero_device_status;-;+zero3_unit_step;-;")


def test_no_tool_attached_costs_nothing_visible(tracer_so):
    """Without an injection library the ranges are no-ops: the same calls return the
    same codes and the tracer records nothing."""
    env = {k: v for k, v in os.environ.items() if k != "NVTX_INJECTION64_PATH"}
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, so=tracer_so)],
                       capture_output=True, text=True, timeout=120, env=env)
    assert r.returncode == 0, r.stderr
    lines = r.stdout.splitlines()
    assert lines[1:] in ([], [""])
