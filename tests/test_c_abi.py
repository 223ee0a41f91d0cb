"""The header is plain C11 and the library is usable from C alone (no Python, no torch)."""
import os
import subprocess

import pytest

from conftest import cuda_available

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIBDIR = os.path.join(ROOT, "zero_partitioned_mixed_adam_gb300")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def demo(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("c") / "abi_demo")
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-O2",
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
                    os.path.join(ROOT, "tests", "c", "abi_demo.c"), "-o", exe,
                    "-L", LIBDIR, "-lzeroadam", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
                    f"-Wl,-rpath,{LIBDIR}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"],
                   check=True)
    return exe


def test_c_program_plans_and_validates(demo):
    r = subprocess.run([demo, "plan"], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert "plan ok" in r.stdout


@pytest.mark.gpu
@pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")
def test_c_program_runs_a_step(demo):
    r = subprocess.run([demo, "step"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "step ok" in r.stdout


@pytest.mark.gpu
@pytest.mark.skipif(not cuda_available(), reason="needs a CUDA GPU")
def test_c_program_runs_a_unit_step(demo):
    r = subprocess.run([demo, "unit"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "unit ok" in r.stdout
