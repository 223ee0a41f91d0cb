"""bench.py's one JSON line: every key the benchmark contract names, for the reference arm
(the oracle on the host cores: runs on CPU) and for the library's arm (on a GPU)."""
import json
import os
import subprocess
import sys

import pytest

from conftest import cuda_available

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e",
        "gpu_launches", "cpu_baseline")


def _line(*args, timeout=600):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                       capture_output=True, text=True, timeout=timeout, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def _common(d, steps, warmup):
    for k in BASE:
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == warmup
    assert d["unit"] == "Gelem/s" and d["higher_is_better"] is True
    assert d["scaling"] == "weak" and d["data"] == "synthetic" and d["vs_baseline"] is None
    assert d["config"]["workload"] == "tiny" and d["value"] > 0 and d["ms_per_step"] > 0
    e = d["e2e"]
    for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert k in e, k


def test_reference_arm_line():
    d = _line("--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3")
    _common(d, 1, 3)
    assert d["impl"] == "reference" and d["gpu_launches"] == 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    c = d["config"]   # the workload's own description, as our arm prints it
    assert c["shard"] == 250_001 and c["bytes_per_step"] == (2 * 4 + 26) * 1_000_003
    assert c["l2"].startswith("L2 flushed before every timed step: a 258 MiB write")


def test_config_describes_the_workload_alone():
    """Both arms build config from the workload: its sizes, the algorithmic bytes of a
    step ((2N + 26) per stepped element, plus 4 per unit element for a ZeRO-3 unit) and
    the L2 handling; nothing in it depends on the implementation that ran."""
    import bench
    cases = {"1p3b": (81_250_000, 58 * 1_300_000_000),
             "7b_rank3": (875_000_000, 42 * 875_000_000),
             "unit:16777216:8": (2_097_152, 4 * 16_777_216 + 42 * 2_097_152),
             "shard:202383360:64": (3_162_240, 154 * 3_162_240)}
    for name, (shard, nbytes) in cases.items():
        c = bench._config(bench._workload(name))
        assert (c["shard"], c["bytes_per_step"]) == (shard, nbytes), name
        assert c["l2"] == "inputs larger than L2 (no flush)"
    assert "unit_step" in bench._config(bench._workload("unit:16777216:8"))


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"],
                       capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert r.returncode != 0


@pytest.mark.gpu
@pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")
def test_our_arm_line():
    d = _line("--workload", "tiny", "--steps", "5", "--warmup", "3", "--cpu-seconds", "1",
              "--e2e-steps", "2")
    _common(d, 5, 3)
    assert "impl" not in d and d["gpu_launches"] == 5
    r = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] == 4 * 2 * 1_000_003
    assert e["d2h_bytes_per_step"] == 2 * 1_000_003
    c = d["clocks"]
    for k in ("sm_mhz", "sm_max_mhz", "reasons"):
        assert k in c, k
    assert d["config"]["l2"].startswith("L2 flushed")   # tiny moves less than 4 L2 sizes
    assert d["launches_per_step"] == ["zero_adam_step_kernel"]
    ref = _line("--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3")
    assert ref["config"] == d["config"]   # both arms describe the same configuration


def test_workload_names():
    """The bench's workload names: the named configurations, a ZeRO-3 unit (its gather and
    rank 0's step) and the same unit's step alone."""
    import bench
    from synth import configs as C
    assert bench._workload("1p3b") is C.B1P3
    assert bench._workload("7b_rank3_prewarm").prewarm == 5
    u = bench._workload("unit:16777216:8")
    s = bench._workload("shard:16777216:8")
    assert u.name.startswith("unit") and not s.name.startswith("unit")
    for w in (u, s):
        assert (w.numel, w.world, w.rank, w.grad_layout, w.param_layout) == \
            (16777216, 8, 0, "shard", "shard")
        assert w.master_spec() == u.master_spec() and w.grad_spec(3, 2) == u.grad_spec(3, 2)
    with pytest.raises(SystemExit):
        bench._workload("nonesuch")


@pytest.mark.gpu
@pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")
@pytest.mark.parametrize("mode", ["fused", "separate"])
def test_unit_workload_line(mode):
    """A ZeRO-3 unit workload's line: one zero3_unit_step call per step (one launch for a
    unit this small) or the gather and the step as two calls; the roofline names the
    dominant launch and the device status is clear."""
    d = _line("--workload", "unit:1048576:8", "--unit-mode", mode, "--steps", "3", "--warmup",
              "3", "--no-e2e", "--no-cpu-baseline")
    assert d["config"]["workload"] == "unit1048576_n8" and d["device_status"] == "ok"
    assert d["value"] > 0 and d["roofline"]["bound"] == "hbm"
    names = [k["kernel"] for k in d["kernels"]]
    if mode == "fused":
        assert names == ["zero3_unit_step_kernel"] and d["gpu_launches"] == 3
    else:
        assert names == ["zero3_unit_gather_tma_kernel", "zero_adam_step_tma_grad_kernel"]
        assert d["gpu_launches"] == 6
    assert d["config"]["bytes_per_step"] == 4 * 1048576 + (2 * 8 + 26) * 131072


@pytest.mark.parametrize("variant,grads,reduce", [("f32", "fp32", "fp32 sum"),
                                                  ("bf16sum", "bf16", "bf16-rounded sum")])
def test_reference_arm_gradient_variants(variant, grads, reduce):
    """The f4 variants reach the oracle: the reference arm steps the same variant."""
    d = _line("--impl", "reference", "--workload", "tiny", "--grad-variant", variant,
              "--steps", "1", "--warmup", "3")
    assert d["config"]["gradients"] == grads and d["config"]["reduce"] == reduce
    assert d["config"]["workload"] == f"tiny+{variant}" and d["value"] > 0
