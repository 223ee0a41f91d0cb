"""The committed DRAM-traffic records bench.py reports beside its roofline: the code hash
that keys them ignores comments but not code, and every record is self-consistent
(bytes per element = (read + write) / elements, within the kernel's algorithmic bytes)."""
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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
            kernel, world = name.split("/N")
            assert kernel.startswith(("zero_adam_step", "zero3_unit_gather")) and int(world) >= 1
            per = (r["dram_read_bytes"] + r["dram_write_bytes"]) / r["elements"]
            assert abs(per - r["dram_bytes_per_element"]) < 1e-4
            # writes still in L2 at the kernel's end make it a little below the algorithmic bytes
            assert 0.85 * r["algorithmic_bytes_per_element"] < per <= 1.02 * r["algorithmic_bytes_per_element"]
            n += 1
    assert n >= 5
