"""The committed DRAM-traffic records bench.py reports beside its roofline: the code hash
that keys them ignores comments but not code, and every record is self-consistent
(bytes per element = (read + write) / elements, within the kernel's algorithmic bytes)."""
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_kernel_source_hash_covers_the_headers(tmp_path):
    """A change in a shared header (where part of a kernel's device code lives) voids
    the kernel's records; a comment change does not."""
    cu = tmp_path / "k.cu"
    cu.write_text("int k() { return f(); }\n")
    h = tmp_path / "ops.h"
    h.write_text("inline int f() { return 1; }\n")
    first = bench.kernel_source_hash(str(cu))
    h.write_text("inline int f() { return 1; }  // note\n")
    assert bench.kernel_source_hash(str(cu)) == first
    h.write_text("inline int f() { return 2; }\n")
    assert bench.kernel_source_hash(str(cu)) != first


def test_code_hash_ignores_comments_not_code(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("int f(int x) {\n  return x + 1;  // one more\n}\n")
    b = tmp_path / "b.cu"
    b.write_text("// header\nint f(int x) {\n\n  return x + 1;   // a different comment\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("int f(int x) {\n  return x + 2;  // one more\n}\n")
    assert bench.code_hash(a) == bench.code_hash(b)
    assert bench.code_hash(a) != bench.code_hash(c)


def test_records_are_consistent():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    n = 0
    for key, kernels in rec.items():
        if key.startswith("_"):
            continue
        assert len(key) == 64
        for name, r in kernels.items():
            kernel, rest = name.split("/N")
            world, _, variant = rest.partition("/")
            assert kernel.startswith(("zero_adam_step", "zero3_unit_gather", "zero3_unit_step"))
            assert int(world) >= 1 and variant in ("", "f32", "bf16sum")
            per = (r["dram_read_bytes"] + r["dram_write_bytes"]) / r["elements"]
            assert abs(per - r["dram_bytes_per_element"]) < 1e-4
            # every input byte is read once: the reads match the algorithmic reads
            reads = r["dram_read_bytes"] / r["elements"]
            alg_r = r["algorithmic_read_bytes_per_element"]
            assert 0.98 * alg_r <= reads <= 1.02 * alg_r, name
            # writes still in L2 at the kernel's end make the total a little below the
            # algorithmic bytes (far below for a launch whose working set is near L2's size)
            alg = r["algorithmic_bytes_per_element"]
            lower = 0.5 if r.get("writes_in_l2") else 0.85
            assert lower * alg < per <= 1.02 * alg, name
            n += 1
    assert n >= 4


def test_traffic_key_names_the_gradient_variant():
    from synth import configs as C
    import dataclasses
    wl = C.WORKLOADS["gpt2"]
    assert bench.traffic_key("zero_adam_step_kernel", wl) == "zero_adam_step_kernel/N8"
    f32 = dataclasses.replace(wl, grad_f32=True)
    s16 = dataclasses.replace(wl, acc_bf16=True)
    assert bench.traffic_key("zero_adam_step_kernel", f32) == "zero_adam_step_kernel/N8/f32"
    assert bench.traffic_key("zero_adam_step_kernel", s16) == "zero_adam_step_kernel/N8/bf16sum"


def test_two_launch_traffic_is_the_sum_of_its_records():
    """A call that launches two kernels (a large unit's gather, then its step) reports the
    sum of the two records; a kernel without a record gives None, not a partial sum."""
    wl = bench._workload("unit:202383360:64")
    S = -(-wl.numel // wl.world)
    g = bench.launch_traffic("zero3_unit_gather_tma_kernel", wl, S)
    st = bench.launch_traffic("zero_adam_step_tma_grad_kernel", wl, S)
    both = bench.launch_traffic("zero3_unit_gather_tma_kernel+zero_adam_step_tma_grad_kernel", wl, S)
    assert g and st and abs(both - (g + st)) < 1.0
    assert bench.launch_traffic("zero3_unit_gather_tma_kernel+no_such_kernel", wl, S) is None
