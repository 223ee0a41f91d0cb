"""The C ABI without a GPU: the library loads, exports what the header declares,
plans layouts exactly as the oracle does, and rejects bad arguments with the
documented status codes before touching CUDA."""
import ctypes
import math
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def za():
    import __graft_entry__
    __graft_entry__.build()
    import zero_partitioned_mixed_adam_gb300 as za
    return za


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "zeroadam.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(zero\w*)\s*\(", text, flags=re.M)))


def test_header_declarations_are_exported(za):
    names = _declared_functions()
    assert set(names) == set(za.EXPORTS), names
    lib = ctypes.CDLL(za.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"


def test_binding_constants_match_the_header(za):
    """Every numeric #define of the header has the same value in the Python binding
    (status codes through za.ERRORS)."""
    text = open(os.path.join(ROOT, "include", "zeroadam.h")).read()
    defines = re.findall(r"^#define (ZERO_\w+)\s+\(?(-?(?:0x[0-9a-fA-F]+|\d+))\)?", text, flags=re.M)
    assert len(defines) >= 25
    errors = {v: k for k, v in za.ERRORS.items()}
    for name, value in defines:
        v = int(value, 0)
        if name.startswith("ZERO_E_"):
            assert errors[name] == v, name
        else:
            assert getattr(za, name) == v, name


def test_library_links_the_shared_cuda_runtime(za):
    with open("/proc/self/maps") as f:
        maps = f.read()
    assert za.LIB_PATH in maps


def test_plan_matches_oracle_brute_force(za):
    for numel in range(1, 201):
        for world in range(1, 18):
            p = za.zero_plan(numel, world)
            o = oracle.plan(numel, world)
            for k in ("numel", "world", "shard", "pad", "padded", "bytes_dp", "bytes_z1",
                      "bytes_z2", "bytes_z3", "state_bytes_rank"):
                assert getattr(p, k) == o[k], (numel, world, k)
            for k in ("formula_dp", "formula_z1", "formula_z2", "formula_z3", "comm_dp",
                      "comm_z1", "comm_z2", "comm_z3"):
                assert math.isclose(getattr(p, k), o[k], rel_tol=1e-14, abs_tol=1e-9), \
                    (numel, world, k)


def test_plan_config_sizes(za):
    for numel, world, shard, pad in ((1_000_003, 4, 250_001, 1), (124_439_808, 8, 15_554_976, 0),
                                     (1_300_000_000, 16, 81_250_000, 0),
                                     (7_000_000_000, 8, 875_000_000, 0),
                                     (202_383_360, 64, 3_162_240, 0)):
        p = za.zero_plan(numel, world)
        assert (p.shard, p.pad) == (shard, pad)


def test_plan_communication_ledger(za):
    """'The three stages' last column and 'Exercises' (second answer): DP's all-reduce
    sends 2(N-1)/N of the bf16 gradients per card, ZeRO-1/2 exactly the same
    (reduce-scatter + all-gather), ZeRO-3 about 1.5 times that."""
    for world in (2, 4, 8, 16, 64):
        numel = 10**9
        p = za.zero_plan(numel, world)
        grad_bytes = 2 * numel
        assert p.comm_dp == pytest.approx(2 * (world - 1) / world * grad_bytes)
        assert p.comm_z1 == p.comm_dp and p.comm_z2 == p.comm_dp
        assert p.comm_z3 / p.comm_dp == pytest.approx(1.5)
    # large N: the all-reduce sends about twice the gradient size ("about 2 x 2 Psi = 4 Psi")
    p = za.zero_plan(10**9, 1024)
    assert p.comm_dp / (4 * 10**9) == pytest.approx(1.0, rel=1e-3)


def test_plan_errors(za):
    with pytest.raises(za.ZeroError) as e:
        za.zero_plan(0, 4)
    assert e.value.code == "ZERO_E_NUMEL"
    with pytest.raises(za.ZeroError) as e:
        za.zero_plan(10, 0)
    assert e.value.code == "ZERO_E_WORLD"
    with pytest.raises(za.ZeroError) as e:
        za.zero_plan(10, za.ZERO_MAX_WORLD + 1)
    assert e.value.code == "ZERO_E_WORLD"
    with pytest.raises(za.ZeroError) as e:
        za.zero_plan(2**62, 1024)
    assert e.value.code == "ZERO_E_NUMEL"
    assert za.raw_lib().zero_plan(10, 2, None) == -1


# Fake device addresses: every call below fails its checks before any CUDA call.
BASE = 1 << 40


def _step(za, plan, rank=-1, grads=None, layout=0, master=BASE + 2**30, m=BASE + 2 * 2**30,
          v=BASE + 3 * 2**30, param=BASE + 4 * 2**30, player=0, lr=1e-3, b1=0.9, b2=0.999,
          eps=1e-8, t=1):
    if grads is None:
        grads = [BASE + 5 * 2**30 + k * 2**28 for k in range(plan.world)]
    ptrs = (ctypes.c_void_p * max(len(grads), 1))(*grads)
    return za.raw_lib().zero_adam_step(ctypes.byref(plan), rank, ptrs, layout, master, m, v,
                                       param, player, lr, b1, b2, eps, t, None)


def test_step_argument_errors(za):
    plan = za.zero_plan(1000, 4)
    lib = za.raw_lib()
    codes = {v: k for k, v in za.ERRORS.items()}
    assert lib.zero_adam_step(None, -1, None, 0, 1, 1, 1, 1, 0, 1e-3, .9, .999, 1e-8, 1,
                              None) == codes["ZERO_E_NULLPTR"]
    assert _step(za, plan, rank=4) == codes["ZERO_E_RANK"]
    assert _step(za, plan, rank=-2) == codes["ZERO_E_RANK"]
    assert _step(za, plan, t=0) == codes["ZERO_E_STEP"]
    assert _step(za, plan, lr=-1.0) == codes["ZERO_E_HPARAM"]
    assert _step(za, plan, lr=float("nan")) == codes["ZERO_E_HPARAM"]
    assert _step(za, plan, b1=1.0) == codes["ZERO_E_HPARAM"]
    assert _step(za, plan, b2=-0.1) == codes["ZERO_E_HPARAM"]
    assert _step(za, plan, eps=float("inf")) == codes["ZERO_E_HPARAM"]
    assert _step(za, plan, layout=3) == codes["ZERO_E_LAYOUT"]
    assert _step(za, plan, layout=1) == codes["ZERO_E_LAYOUT"]      # shard grads, all ranks
    assert _step(za, plan, player=1) == codes["ZERO_E_LAYOUT"]      # shard params, all ranks
    assert _step(za, plan, master=0) == codes["ZERO_E_NULLPTR"]
    assert _step(za, plan, grads=[BASE, 0, BASE + 2**20, BASE + 2**21]) == codes["ZERO_E_NULLPTR"]
    assert _step(za, plan, master=BASE + 2**30 + 2) == codes["ZERO_E_ALIGN"]
    assert _step(za, plan, param=BASE + 4 * 2**30 + 1) == codes["ZERO_E_ALIGN"]
    assert _step(za, plan, m=BASE + 2**30 + 400) == codes["ZERO_E_ALIAS"]   # m overlaps master
    g = [BASE + 5 * 2**30 + k * 2**28 for k in range(4)]
    assert _step(za, plan, grads=g, param=g[2] + 100) == codes["ZERO_E_ALIAS"]
    bad = za.zero_plan(1000, 4)
    bad.shard = 251
    assert _step(za, bad) == codes["ZERO_E_PLAN"]
    bad = za.zero_plan(1000, 4)
    bad.world = 0
    assert _step(za, bad) == codes["ZERO_E_WORLD"]
    # single rank owning no real element: valid, nothing to do, no CUDA call
    empty = za.zero_plan(9, 4)   # shard 3: rank 3 owns [9, 12), all padding
    assert _step(za, empty, rank=3, layout=1, player=1) == 0


def test_pointer_array_is_marshalled_once(za):
    """A PointerArray carries the C array of addresses built when it was made; the calls
    pass that array itself, and check its length against the plan like a list's."""
    addrs = [BASE + 5 * 2**30 + k * 2**28 for k in range(4)]
    pa = za.pointer_array(addrs)
    assert len(pa) == 4 and list(pa.buffers) == addrs
    assert za._ptrs(pa) is pa.arr
    assert [pa.arr[k] for k in range(4)] == addrs
    fresh = za._ptrs(addrs)
    assert fresh is not pa.arr and [fresh[k] for k in range(4)] == addrs
    plan = za.zero_plan(1000, 4)
    kw = dict(lr=1e-3, t=0)
    # t = 0 is refused before any CUDA call: the same error through a list and the array
    for grads in (addrs, pa):
        with pytest.raises(za.ZeroError) as e:
            za.zero_adam_step(plan, -1, grads, BASE + 2**30, BASE + 2 * 2**30, BASE + 3 * 2**30,
                              BASE + 4 * 2**30, **kw)
        assert e.value.code == "ZERO_E_STEP"
    with pytest.raises(ValueError):
        za.zero_adam_step(za.zero_plan(1000, 3), -1, pa, BASE + 2**30, BASE + 2 * 2**30,
                          BASE + 3 * 2**30, BASE + 4 * 2**30, **kw)
    with pytest.raises(ValueError):
        za.zero3_unit_gather(za.zero_plan(1000, 2), pa, BASE + 2**30)


def test_range_argument_errors(za):
    plan = za.zero_plan(1000, 4)
    lib = za.raw_lib()
    codes = {v: k for k, v in za.ERRORS.items()}
    g = [BASE + 5 * 2**30 + k * 2**28 for k in range(4)]
    ptrs = (ctypes.c_void_p * 4)(*g)

    def rng(begin, end, layout=2, rank=-1, player=0, master=BASE + 2**30):
        return lib.zero_adam_step_range(ctypes.byref(plan), rank, begin, end, ptrs, layout,
                                        master, BASE + 2 * 2**30, BASE + 3 * 2**30,
                                        BASE + 4 * 2**30, player, 1e-3, .9, .999, 1e-8, 1, None)

    assert rng(-1, 10) == codes["ZERO_E_RANGE"]
    assert rng(20, 10) == codes["ZERO_E_RANGE"]
    assert rng(0, 10, layout=3) == codes["ZERO_E_LAYOUT"]
    assert rng(0, 10, layout=0x40) == codes["ZERO_E_LAYOUT"]            # unknown flag
    assert rng(0, 10, master=BASE + 2**30 + 2) == codes["ZERO_E_ALIGN"]
    # fp32 gradients must be 4-byte aligned
    ptrs2 = (ctypes.c_void_p * 4)(*[x + 2 for x in g])
    assert lib.zero_adam_step_range(ctypes.byref(plan), -1, 0, 10, ptrs2, 2 | 0x10,
                                    BASE + 2**30, BASE + 2 * 2**30, BASE + 3 * 2**30,
                                    BASE + 4 * 2**30, 0, 1e-3, .9, .999, 1e-8, 1,
                                    None) == codes["ZERO_E_ALIGN"]
    # windows that hold none of the stepped rank's elements: valid, nothing launched
    assert rng(0, 0) == 0
    assert rng(2000, 3000) == 0
    assert rng(0, 100, rank=2) == 0        # rank 2 owns [500, 750)
    # zero_adam_step itself has no window layout
    assert _step(za, plan, layout=2) == codes["ZERO_E_LAYOUT"]


def test_gather_argument_errors(za):
    plan = za.zero_plan(1000, 4)
    lib = za.raw_lib()
    codes = {v: k for k, v in za.ERRORS.items()}
    shards = [BASE + k * 2**20 for k in range(4)]
    ptrs = (ctypes.c_void_p * 4)(*shards)
    assert lib.zero3_unit_gather(ctypes.byref(plan), ptrs, None, None) == codes["ZERO_E_NULLPTR"]
    assert lib.zero3_unit_gather(ctypes.byref(plan), None, BASE + 2**30,
                                 None) == codes["ZERO_E_NULLPTR"]
    assert lib.zero3_unit_gather(ctypes.byref(plan), ptrs, BASE + 2**30 + 1,
                                 None) == codes["ZERO_E_ALIGN"]
    assert lib.zero3_unit_gather(ctypes.byref(plan), ptrs, shards[1] - 10,
                                 None) == codes["ZERO_E_ALIAS"]


def test_unit_step_argument_errors(za):
    """zero3_unit_step checks both parts as their own calls do, and that the parts'
    buffers are disjoint (they run side by side); every error is found on the host,
    before any CUDA call, so these fake addresses are never touched."""
    plan = za.zero_plan(1000, 4)          # shard 250
    lib = za.raw_lib()
    codes = {v: k for k, v in za.ERRORS.items()}
    shards = [BASE + k * 2**20 for k in range(4)]
    grads = [BASE + 5 * 2**30 + k * 2**28 for k in range(4)]
    W, M, V, P, FULL = (BASE + 2**30, BASE + 2 * 2**30, BASE + 3 * 2**30, BASE + 4 * 2**30,
                        BASE + 6 * 2**30)

    def call(rank=1, full=FULL, sh=shards, g=grads, master=W, param=P, layout=1, player=1,
             t=1, p=plan):
        sp = (ctypes.c_void_p * 4)(*sh)
        gp = (ctypes.c_void_p * 4)(*g)
        return lib.zero3_unit_step(ctypes.byref(p) if p is not None else None, rank, sp, full,
                                   gp, layout, master, M, V, param, player, 1e-3, .9, .999,
                                   1e-8, t, None)

    assert call(p=None) == codes["ZERO_E_NULLPTR"]
    assert call(full=0) == codes["ZERO_E_NULLPTR"]
    assert call(rank=4) == codes["ZERO_E_RANK"]
    assert call(t=0) == codes["ZERO_E_STEP"]
    assert call(layout=2) == codes["ZERO_E_LAYOUT"]          # no window layout
    assert call(full=FULL + 1) == codes["ZERO_E_ALIGN"]
    assert call(full=shards[2] + 16) == codes["ZERO_E_ALIAS"]   # the gather's own check
    assert call(full=P - 100) == codes["ZERO_E_ALIAS"]          # unit over the step's params
    assert call(full=grads[3] + 64) == codes["ZERO_E_ALIAS"]    # unit over a gradient
    assert call(param=shards[1] + 2) == codes["ZERO_E_ALIAS"]   # a step output over a shard
    assert call(master=shards[3]) == codes["ZERO_E_ALIAS"]


def test_gather_rows_argument_errors(za):
    lib = za.raw_lib()
    codes = {v: k for k, v in za.ERRORS.items()}
    shards = [BASE + k * 2**20 for k in range(4)]
    ptrs = (ctypes.c_void_p * 4)(*shards)

    def call(rows, cols, world=4, full=BASE + 2**30, p=ptrs, n=None):
        n = len(rows) if n is None else n
        r = (ctypes.c_int64 * max(1, len(rows)))(*rows)
        c = (ctypes.c_int64 * max(1, len(cols)))(*cols)
        return lib.zero3_unit_gather_rows(n, r, c, world, p, full, None)

    assert call([10], [3], n=0) == codes["ZERO_E_SHAPE"]
    assert call([10] * 257, [3] * 257) == codes["ZERO_E_SHAPE"]
    assert call([10, 0], [3, 3]) == codes["ZERO_E_SHAPE"]
    assert call([10, 5], [3, -1]) == codes["ZERO_E_SHAPE"]
    assert call([2**40], [2**40]) == codes["ZERO_E_SHAPE"]
    assert call([10], [3], world=0) == codes["ZERO_E_WORLD"]
    assert call([10], [3], full=0) == codes["ZERO_E_NULLPTR"]
    assert call([10], [3], full=BASE + 2**30 + 1) == codes["ZERO_E_ALIGN"]
    assert call([10], [3], full=shards[2] + 4) == codes["ZERO_E_ALIAS"]
    bad = (ctypes.c_void_p * 4)(shards[0], None, shards[2], shards[3])
    assert call([10], [3], p=bad) == codes["ZERO_E_NULLPTR"]
    assert za.rows_layout([(10, 3), (7, 2)], 4) == (3 * 3 + 2 * 2, 44)


def test_device_status_without_a_gpu(za):
    # no CUDA device in this process: the call reports it instead of failing
    if not __import__("conftest").cuda_available():
        assert za.device_status() == -12


def test_strerror(za):
    for code in za.ERRORS:
        s = za.strerror(code)
        assert s and s != "unknown status"
    assert za.strerror(0) == "ok"
    assert za.version() == 0x000100


def test_test_hook_is_off_without_its_environment_variable():
    """zero_test_withhold_copies answers only when ZEROADAM_TEST_HOOKS=1: a process
    without it gets ZERO_E_HOOK and the flag stays off; with it the call sets the flag
    and returns the previous setting.  Host only (the flag is read at launch time)."""
    import subprocess
    import sys
    child = ("import sys; sys.path.insert(0, %r)\n"
             "import zero_partitioned_mixed_adam_gb300 as za\n"
             "lib = za.raw_lib()\n"
             "print(lib.zero_test_withhold_copies(1), lib.zero_test_withhold_copies(0))\n" % ROOT)
    base = {k: v for k, v in os.environ.items() if k != "ZEROADAM_TEST_HOOKS"}
    for env, want in ((base, "-16 -16"), (dict(base, ZEROADAM_TEST_HOOKS="0"), "-16 -16"),
                      (dict(base, ZEROADAM_TEST_HOOKS="1"), "0 1")):
        r = subprocess.run([sys.executable, "-c", child], capture_output=True, text=True,
                           timeout=120, env=env)
        assert r.returncode == 0, r.stderr
        assert r.stdout.split()[-2:] == want.split(), (env.get("ZEROADAM_TEST_HOOKS"), r.stdout)
