"""Pins of the oracle to things other than itself (CPU only).

Each test checks the oracle against what the pages print, against closed forms
of the mathematics, against invariants of the method, or against an
independent library routine (torch.optim.Adam, torch's bf16 cast, numpy
concatenation).  A dropped term, a wrong sign or index, a swapped beta or a
missing average fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

LR, B1, B2, EPS = 1e-3, 0.9, 0.999, 1e-8


def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ planner


def test_plan_brute_force_layout():
    """shard = ceil(numel/world); the N ranges tile [0, N*shard) disjointly; pad < N."""
    for numel in range(1, 201):
        for world in range(1, 18):
            p = oracle.plan(numel, world)
            S = p["shard"]
            assert S * world >= numel and (S - 1) * world < numel
            assert p["padded"] == S * world
            assert 0 <= p["pad"] < world and p["pad"] == S * world - numel
            owner = np.full(p["padded"], -1)
            for r in range(world):
                assert (owner[r * S:(r + 1) * S] == -1).all()
                owner[r * S:(r + 1) * S] = r
            assert (owner >= 0).all()
            # every real element is owned by exactly one rank; the pad sits at the end
            assert (np.arange(p["padded"]) // S == owner).all()


def test_plan_bytes_equal_table_when_divisible_and_exceed_by_padding_otherwise():
    """Integer bytes = the table's formulas when N | Psi, else formula + c*pad/N (c=12,14,16)."""
    for numel in range(1, 201):
        for world in range(1, 18):
            p = oracle.plan(numel, world)
            P, N, pad = numel, world, p["pad"]
            assert p["bytes_dp"] == 16 * P
            assert math.isclose(p["formula_dp"], 16 * P)
            # the table's rational expressions, evaluated independently here
            assert math.isclose(p["formula_z1"], 4 * P + 12 * P / N, rel_tol=1e-15)
            assert math.isclose(p["formula_z2"], 2 * P + 14 * P / N, rel_tol=1e-15)
            assert math.isclose(p["formula_z3"], 16 * P / N, rel_tol=1e-15)
            for key, c in (("z1", 12), ("z2", 14), ("z3", 16)):
                extra = p[f"bytes_{key}"] - (4 * P if key == "z1" else 2 * P if key == "z2" else 0)
                # partitioned components hold c bytes per shard element
                assert extra == c * p["shard"]
                assert math.isclose(p[f"bytes_{key}"] - p[f"formula_{key}"], c * pad / N,
                                    abs_tol=1e-9)
            assert p["state_bytes_rank"] == 12 * p["shard"]


def test_plan_13b_on_16_cards_exercise(golden_dir):
    g = _golden(golden_dir, "memory_ledger.json")["exercise_13b_16_cards"]
    p = oracle.plan(g["numel"], g["world"])
    assert p["pad"] == 0
    assert p["bytes_z1"] / 1e9 == pytest.approx(g["zero1_gb"], abs=1e-12)
    assert p["bytes_z2"] / 1e9 == pytest.approx(g["zero2_gb_exact"], abs=1e-12)
    assert round(p["bytes_z2"] / 1e9, 1) == g["zero2_gb_printed"]
    assert p["bytes_z3"] / 1e9 == pytest.approx(g["zero3_gb"], abs=1e-12)
    left = {s: g["card_gb"] - p[f"bytes_{s}"] / 1e9 for s in ("dp", "z1", "z2", "z3")}
    first = next(s for s in ("dp", "z1", "z2", "z3") if left[s] >= g["activation_budget_gb"])
    assert {"z2": "ZeRO-2"}[first] == g["first_stage_leaving_budget"]


def test_plan_16_bytes_and_12_bytes_of_optimizer_state(golden_dir):
    g = _golden(golden_dir, "memory_ledger.json")
    p = oracle.plan(1000, 1)
    assert p["bytes_dp"] == g["bytes_per_param_dp"]["value"] * 1000
    # with one card nothing is partitioned: every stage is plain DP
    assert p["bytes_z1"] == p["bytes_z2"] == p["bytes_z3"] == p["bytes_dp"]
    # what ZeRO-1 partitions is the optimizer state: DP - Z1 at large N -> 12 B/param
    q = oracle.plan(10**6 * 4096, 4096)
    per_param = (q["bytes_dp"] - q["bytes_z1"]) / q["numel"]
    assert per_param == pytest.approx(g["optimizer_state_bytes_per_param"]["value"], rel=1e-3)


def test_plan_stage_reduction_limits(golden_dir):
    g = _golden(golden_dir, "memory_ledger.json")["stage_reduction_limits"]
    p = oracle.plan(10**12, 10**6)
    assert p["bytes_dp"] / p["bytes_z1"] == pytest.approx(g["zero1"], rel=1e-5)
    assert p["bytes_dp"] / p["bytes_z2"] == pytest.approx(g["zero2"], rel=1e-5)
    # and the reductions grow monotonically toward those limits
    prev1 = prev2 = 0.0
    for n in (1, 2, 4, 8, 64, 1024):
        q = oracle.plan(2**30, n)
        r1, r2 = q["bytes_dp"] / q["bytes_z1"], q["bytes_dp"] / q["bytes_z2"]
        assert prev1 < r1 < g["zero1"] and prev2 < r2 < g["zero2"] or n == 1
        prev1, prev2 = r1, r2


def test_plan_optimizer_state_8x_at_8_gpus(golden_dir):
    g = _golden(golden_dir, "memory_ledger.json")["optimizer_state_8_gpus"]
    p1 = oracle.plan(8 * 10**9, 1)
    p8 = oracle.plan(8 * 10**9, g["world"])
    assert p1["state_bytes_rank"] / p8["state_bytes_rank"] == g["reduction"]


def test_plan_demo_mlp(golden_dir):
    g = _golden(golden_dir, "memory_ledger.json")["demo_mlp"]
    numel = sum(i * o + o for i, o in g["layers"])  # weights + biases of each Linear
    assert numel == g["numel"]
    p = oracle.plan(numel, g["world"])
    assert p["shard"] == g["shard"]
    assert p["state_bytes_rank"] == g["state_bytes_rank"]
    full = 3 * numel * 4
    assert full == g["full_state_bytes"]
    assert round(full / p["state_bytes_rank"]) == g["printed_ratio"]


def test_plan_communication_ledger(golden_dir):
    g = _golden(golden_dir, "memory_ledger.json")["communication"]
    for world in (1, 2, 3, 8, 16, 64):
        for numel in (12, 1000, 10**9):
            p = oracle.plan(numel, world)
            grad_bytes = 2 * p["padded"]
            assert p["comm_dp"] == pytest.approx(2 * (world - 1) / world * grad_bytes, rel=1e-15)
            assert p["comm_z1"] / max(p["comm_dp"], 1e-300) == pytest.approx(g["zero12_vs_dp"]) \
                or world == 1
            assert p["comm_z2"] == p["comm_z1"]
            if world > 1:
                assert p["comm_z3"] / p["comm_dp"] == pytest.approx(g["zero3_vs_dp"], rel=1e-15)
            else:
                assert p["comm_dp"] == p["comm_z3"] == 0.0
    big = oracle.plan(10**12, 10**6)
    assert big["comm_dp"] / big["numel"] == pytest.approx(g["dp_large_n_bytes_per_param"],
                                                          rel=1e-5)


def test_plan_rejects_bad_arguments():
    for numel, world in ((0, 1), (-5, 2), (10, 0), (10, -1)):
        with pytest.raises(ValueError):
            oracle.plan(numel, world)


# ------------------------------------------------------------------ bf16 cast


def _torch_bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_cast_matches_torch_exhaustive_low_halves():
    """Every low half-word under high halves covering zero, denormals, ties, carries, max, inf."""
    highs = np.array([0x0000, 0x0001, 0x007f, 0x0080, 0x3f80, 0x3f81, 0x3fff, 0x4000, 0x7f7f,
                      0x7f7e, 0x8000, 0x8001, 0xbf80, 0xc2c8, 0xff7f, 0x0100, 0x33d6],
                     dtype=np.uint32)
    lows = np.arange(1 << 16, dtype=np.uint32)
    bits = (highs[:, None] << 16 | lows[None, :]).ravel()
    x = bits.view(np.float32)
    assert (oracle.f32_to_bf16(x) == _torch_bf16_bits(x)).all()


def test_bf16_cast_matches_torch_random_and_nan():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    ours = oracle.f32_to_bf16(x)
    ref = _torch_bf16_bits(x)
    nan = np.isnan(x)
    assert (ours[~nan] == ref[~nan]).all()
    # NaN stays NaN (payload bits are not part of the contract)
    assert np.isnan(oracle.bf16_to_f32(ours[nan])).all()


def test_bf16_widening_exact():
    h = np.arange(1 << 16, dtype=np.uint16)
    f = oracle.bf16_to_f32(h)
    ref = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    same = (f.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(f) & np.isnan(ref))
    assert same.all()


# ---------------------------------------------------------- step: special cases


def _bf16(vals):
    return oracle.f32_to_bf16(np.asarray(vals, dtype=np.float32))


def _one_step(grads_rows, master, m=None, v=None, lr=LR, b1=B1, b2=B2, eps=EPS, t=1):
    """Run the oracle's all-ranks step on N rows of bf16 grads of equal length."""
    world = len(grads_rows)
    numel = len(master)
    p = oracle.plan(numel, world)
    grads = []
    for row in grads_rows:
        g = np.zeros(p["padded"], dtype=np.uint16)
        g[:numel] = row
        grads.append(g)
    W = np.zeros(p["padded"], np.float32)
    W[:numel] = master
    M = np.zeros(p["padded"], np.float32)
    V = np.zeros(p["padded"], np.float32)
    if m is not None:
        M[:numel] = m
    if v is not None:
        V[:numel] = v
    par = np.zeros(numel, np.uint16)
    oracle.zero_step(numel, world, -1, grads, W, M, V, par, lr, b1, b2, eps, t)
    return W[:numel], M[:numel], V[:numel], par


def test_reduce_order_is_rank_order_fp32():
    """1 + 2^-24 + 2^-24 summed left to right stays 1 (each add ties to even);
    any other grouping gives 1 + 2^-23.  With beta1 = 0, m after one step is the
    averaged gradient itself."""
    tiny = 2.0**-24
    w0 = np.zeros(1, np.float32)
    # ranks (1, tiny, tiny): acc stays exactly 1.0, g = RN(1/3)
    _, m, _, _ = _one_step([_bf16([1.0]), _bf16([tiny]), _bf16([tiny])], w0, b1=0.0, b2=0.0)
    assert m[0] == np.float32(1.0) / np.float32(3.0)
    # ranks (tiny, tiny, 1): acc = 2^-23 then 1 + 2^-23 exactly
    _, m2, _, _ = _one_step([_bf16([tiny]), _bf16([tiny]), _bf16([1.0])], w0, b1=0.0, b2=0.0)
    assert m2[0] == np.float32(1.0 + 2.0**-23) / np.float32(3.0)
    assert m[0] != m2[0]


def test_average_divides_by_world():
    """Constant gradient c on every rank averages to exactly c; a gradient on one rank only
    averages to c/N (exact for powers of two)."""
    w0 = np.zeros(4, np.float32)
    for world in (1, 2, 3, 4, 8, 16):
        c = np.float32(0.375)
        rows = [_bf16([c, c, -c, 0.0])] * world
        _, m, _, _ = _one_step(rows, w0, b1=0.0, b2=0.0)
        assert (m == np.array([c, c, -c, 0.0], np.float32)).all()
    for world in (2, 4, 8, 16, 64):
        rows = [_bf16([0.5, 0, 0, 0])] + [_bf16([0, 0, 0, 0])] * (world - 1)
        _, m, _, _ = _one_step(rows, w0, b1=0.0, b2=0.0)
        assert m[0] == np.float32(0.5 / world)


def test_first_step_from_zero_state_is_sign_like():
    """t = 1, m = v = 0: m_hat = g and v_hat = g^2 up to rounding, so
    w1 = w0 - lr * g / (|g| + eps), i.e. about w0 - lr*sign(g) for |g| >> eps."""
    rng = np.random.default_rng(1)
    numel, world = 1000, 4
    rows = [_bf16(rng.normal(0, 1e-3, numel)) for _ in range(world)]
    w0 = rng.normal(0, 0.02, numel).astype(np.float32)
    w1, m, v, par = _one_step(rows, w0)
    g = sum(oracle.bf16_to_f32(r).astype(np.float64) for r in rows) / world
    nz = np.abs(g) > 1e-6
    expect = w0.astype(np.float64) - LR * g / (np.abs(g) + EPS)
    assert np.allclose(w1[nz], expect[nz], rtol=3e-7, atol=2e-9)  # fp32 rounding of w
    assert np.allclose(m, (1 - B1) * g, rtol=1e-6, atol=1e-15)
    assert np.allclose(v, (1 - B2) * g * g, rtol=1e-6, atol=1e-20)
    # the sign of the move is opposite to the gradient
    assert (np.sign(w1 - w0)[nz] == -np.sign(g[nz])).all()


def test_zero_gradient_leaves_state_unchanged():
    w0 = np.random.default_rng(2).normal(0, 0.02, 257).astype(np.float32)
    rows = [np.zeros(257, np.uint16)] * 3
    w1, m, v, par = _one_step(rows, w0)
    assert (w1.view(np.uint32) == w0.view(np.uint32)).all()
    assert (m == 0).all() and (v == 0).all()
    assert (par == oracle.f32_to_bf16(w0)).all()


def test_constant_gradient_closed_form_over_steps():
    """Constant gradient c: m_t = (1-b1^t) c, v_t = (1-b2^t) c^2, so every step moves
    w by lr * c / (|c| + eps)."""
    c = 2.0**-10
    world, numel, T = 4, 16, 5
    rows = [_bf16([c] * numel)] * world
    p = oracle.plan(numel, world)
    grads = [np.pad(r, (0, p["padded"] - numel)) for r in rows]
    W = np.full(p["padded"], 0.5, np.float32)
    W[numel:] = 0
    M = np.zeros(p["padded"], np.float32)
    V = np.zeros(p["padded"], np.float32)
    par = np.zeros(numel, np.uint16)
    for t in range(1, T + 1):
        oracle.zero_step(numel, world, -1, grads, W, M, V, par, LR, B1, B2, EPS, t)
        assert np.allclose(M[:numel], (1 - B1**t) * c, rtol=3e-7)
        assert np.allclose(V[:numel], (1 - B2**t) * c * c, rtol=3e-6)
        assert np.allclose(W[:numel], 0.5 - t * LR * c / (c + EPS), rtol=0, atol=3e-8)


def test_eps_sits_outside_the_sqrt():
    """With a large eps the placement matters: w1 = w0 - lr*g/(|g|+eps)."""
    g = 1e-4
    eps = 1e-2
    w1, _, _, _ = _one_step([_bf16([g])], np.zeros(1, np.float32), eps=eps)
    gb = float(oracle.bf16_to_f32(_bf16([g]))[0])
    assert w1[0] == pytest.approx(-LR * gb / (gb + eps), rel=1e-6)
    assert w1[0] != pytest.approx(-LR * gb / math.sqrt(gb * gb + eps), rel=1e-3)


def test_bias_correction_uses_step_number():
    """With m_{t-1}, v_{t-1} = 0 but t = 3, m_hat = (1-b1) g / (1-b1^3)."""
    g = 2.0**-8
    _, m, v, _ = _one_step([_bf16([g])], np.zeros(1, np.float32), t=3, eps=0.0, lr=1.0)
    w1, _, _, _ = _one_step([_bf16([g])], np.zeros(1, np.float32), t=3, eps=0.0, lr=1.0)
    mh = (1 - B1) * g / (1 - B1**3)
    vh = (1 - B2) * g * g / (1 - B2**3)
    assert w1[0] == pytest.approx(-mh / math.sqrt(vh), rel=1e-6)


def test_step_rejects_t_zero():
    p = oracle.plan(4, 1)
    g = [np.zeros(4, np.uint16)]
    z = np.zeros(4, np.float32)
    with pytest.raises(ValueError):
        oracle.zero_step(4, 1, -1, g, z.copy(), z.copy(), z.copy(), np.zeros(4, np.uint16),
                         LR, B1, B2, EPS, 0)


# ------------------------------------------------- step: against torch.optim.Adam


@pytest.mark.parametrize("numel,world,steps", [(19210, 4, 3), (1000, 3, 5), (4097, 8, 3)])
def test_matches_torch_adam_on_the_averaged_gradient(numel, world, steps):
    """The page's own bar: ZeroAdam across ranks vs single-process torch.optim.Adam,
    max |diff| < 1e-5 after 3 steps.  We also hold fp32 state to ~1e-6 relative."""
    rng = np.random.default_rng(numel + world)
    p = oracle.plan(numel, world)
    w0 = rng.normal(0, 0.02, numel).astype(np.float32)
    W = np.zeros(p["padded"], np.float32)
    W[:numel] = w0
    M = np.zeros_like(W)
    V = np.zeros_like(W)
    par = np.zeros(numel, np.uint16)
    ref = torch.nn.Parameter(torch.from_numpy(w0.copy()))
    opt = torch.optim.Adam([ref], lr=LR, betas=(B1, B2), eps=EPS, foreach=False, fused=False)
    for t in range(1, steps + 1):
        rows = [_bf16(rng.normal(0, 1e-3, numel)) for _ in range(world)]
        grads = [np.pad(r, (0, p["padded"] - numel)) for r in rows]
        oracle.zero_step(numel, world, -1, grads, W, M, V, par, LR, B1, B2, EPS, t)
        acc = oracle.bf16_to_f32(rows[0]).copy()
        for r in rows[1:]:
            acc = acc + oracle.bf16_to_f32(r)
        ref.grad = torch.from_numpy(acc / np.float32(world))
        opt.step()
    st = opt.state[ref]
    w_ref = ref.detach().numpy()
    assert np.abs(W[:numel] - w_ref).max() < 1e-5
    assert np.allclose(W[:numel], w_ref, rtol=1e-6, atol=2e-9)
    # torch forms m with lerp, a different rounding path: near-cancelled moments get an
    # absolute floor of 1e-6 of the moment's scale
    m_ref, v_ref = st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()
    assert np.allclose(M[:numel], m_ref, rtol=1e-6, atol=1e-6 * np.abs(m_ref).max())
    assert np.allclose(V[:numel], v_ref, rtol=1e-6, atol=1e-6 * np.abs(v_ref).max())
    assert (par == oracle.f32_to_bf16(W[:numel])).all()


# --------------------------------------------------------- step: invariants


@pytest.mark.parametrize("numel,world", [(1, 1), (7, 3), (37, 5), (1000, 4), (1001, 8), (3, 16)])
def test_sharded_equals_unsharded_bitwise(numel, world):
    """ZeRO changes where state lives, not what is computed: the per-rank sharded
    step equals plain DP Adam on the averaged gradient, bit for bit, every step."""
    rng = np.random.default_rng(numel * 31 + world)
    p = oracle.plan(numel, world)
    w0 = rng.normal(0, 0.02, numel).astype(np.float32)
    Wz = np.zeros(p["padded"], np.float32)
    Wz[:numel] = w0
    Mz, Vz = np.zeros_like(Wz), np.zeros_like(Wz)
    pz = np.zeros(numel, np.uint16)
    Wd, Md, Vd = w0.copy(), np.zeros(numel, np.float32), np.zeros(numel, np.float32)
    pd = np.zeros(numel, np.uint16)
    # per-rank arrays for the single-rank form (each rank owns only its shard)
    S = p["shard"]
    Wr = [Wz[r * S:(r + 1) * S].copy() for r in range(world)]
    Mr = [np.zeros(S, np.float32) for _ in range(world)]
    Vr = [np.zeros(S, np.float32) for _ in range(world)]
    pr = np.zeros(numel, np.uint16)
    for t in range(1, 4):
        rows = [_bf16(rng.normal(0, 1e-3, numel)) for _ in range(world)]
        grads = [np.pad(r, (0, p["padded"] - numel)) for r in rows]
        oracle.zero_step(numel, world, -1, grads, Wz, Mz, Vz, pz, LR, B1, B2, EPS, t)
        oracle.dp_step(numel, world, rows, Wd, Md, Vd, pd, LR, B1, B2, EPS, t)
        for r in range(world):
            oracle.zero_step(numel, world, r, grads, Wr[r], Mr[r], Vr[r], pr, LR, B1, B2, EPS, t,
                             state_base=r * S)
        for a, b in ((Wz[:numel], Wd), (Mz[:numel], Md), (Vz[:numel], Vd)):
            assert (a.view(np.uint32) == b.view(np.uint32)).all()
        assert (pz == pd).all() and (pr == pd).all()
        assert (np.concatenate(Wr).view(np.uint32) == Wz.view(np.uint32)).all()
        assert (np.concatenate(Mr).view(np.uint32) == Mz.view(np.uint32)).all()


def test_padding_tail_never_read_or_written():
    """Indices >= numel are the zero pad: their state stays as it was and the
    parameter buffer beyond numel is not written, whatever the pad's gradient holds."""
    numel, world = 10, 4  # shard 3, pad 2
    p = oracle.plan(numel, world)
    assert p["pad"] == 2
    rng = np.random.default_rng(3)
    grads = [rng.integers(0, 2**16, p["padded"], dtype=np.uint64).astype(np.uint16)
             for _ in range(world)]
    for g in grads:
        g[:numel] = _bf16(rng.normal(0, 1e-3, numel))
    W = np.zeros(p["padded"], np.float32)
    M = np.zeros_like(W)
    V = np.zeros_like(W)
    W[:numel] = rng.normal(0, 0.02, numel)
    par = np.full(p["padded"], 0xABCD, np.uint16)
    oracle.zero_step(numel, world, -1, grads, W, M, V, par, LR, B1, B2, EPS, 1)
    assert (W[numel:] == 0).all() and (M[numel:] == 0).all() and (V[numel:] == 0).all()
    assert (par[numel:] == 0xABCD).all()
    assert (par[:numel] != 0xABCD).all()


def test_window_equals_whole():
    """A window [i0, i1) of the step equals the same indices of the whole step
    (the step is elementwise), including across a shard boundary."""
    numel, world = 1003, 4
    rng = np.random.default_rng(4)
    p = oracle.plan(numel, world)
    grads = [np.pad(_bf16(rng.normal(0, 1e-3, numel)), (0, p["padded"] - numel))
             for _ in range(world)]
    W = np.zeros(p["padded"], np.float32)
    W[:numel] = rng.normal(0, 0.02, numel)
    M, V = np.zeros_like(W), np.zeros_like(W)
    W2, M2, V2 = W.copy(), M.copy(), V.copy()
    par, par2 = np.zeros(numel, np.uint16), np.zeros(numel, np.uint16)
    oracle.zero_step(numel, world, -1, grads, W, M, V, par, LR, B1, B2, EPS, 1)
    i0, i1 = 240, 270  # crosses the rank-0/rank-1 boundary at 251
    win = [g[i0:i1].copy() for g in grads]
    w, m, v, pw = W2[i0:i1].copy(), M2[i0:i1].copy(), V2[i0:i1].copy(), par2[i0:i1].copy()
    oracle.zero_step(numel, world, -1, win, w, m, v, pw, LR, B1, B2, EPS, 1, i0=i0, i1=i1,
                     grad_base=i0, state_base=i0, param_base=i0)
    assert (w.view(np.uint32) == W[i0:i1].view(np.uint32)).all()
    assert (pw == par[i0:i1]).all()


def test_scalars_rounded_once_from_double():
    s = oracle.scalars(1e-3, 0.9, 0.999, 1e-8, 3, 16)
    assert s["omb1"] == np.float32(1.0 - 0.9)       # not 1.0f - 0.9f
    assert s["omb1"] != np.float32(1.0) - np.float32(0.9)
    assert s["bc2"] == np.float32(1.0 - 0.999**3)
    assert s["world"] == 16.0


# ------------------------------------------------------------------ unit gather


def test_unit_gather_brute_force():
    rng = np.random.default_rng(5)
    for U in range(1, 101):
        for N in range(1, 10):
            S = -(-U // N)
            shards = [rng.integers(0, 2**16, S, dtype=np.uint64).astype(np.uint16)
                      for _ in range(N)]
            full = oracle.unit_gather(U, N, shards)
            assert (full == np.concatenate(shards)[:U]).all()


# ------------------------------------------------------- synthetic input recipe


def test_synth_distributions():
    """The input generator draws what the recipe says (moments, zero mask, outliers)."""
    n = 400_000
    x = synth.fill_host(synth.Spec(seed=0, stream=1, sigma=0.02), 0, n, synth.OUT_F32)
    assert abs(x.mean()) < 3 * 0.02 / math.sqrt(n) * 2 and x.std() == pytest.approx(0.02, rel=0.01)
    z = synth.fill_host(synth.Spec(seed=0, stream=2, sigma=1e-3, zero_frac=0.1), 0, n,
                        synth.OUT_BF16)
    z2 = synth.fill_host(synth.Spec(seed=0, stream=2, rank=5, sigma=1e-3, zero_frac=0.1), 0, n,
                         synth.OUT_BF16)
    assert (z == 0).mean() == pytest.approx(0.1, abs=0.003)
    assert ((z == 0) == (z2 == 0)).all()          # the mask is shared by the ranks
    assert not (z == z2).all()
    t3 = synth.fill_host(synth.Spec(seed=0, stream=3, dist=synth.STUDENT_T3, sigma=1.0), 0, n,
                         synth.OUT_F32)
    assert np.median(np.abs(t3)) == pytest.approx(0.7649, abs=0.01)  # median |t_3|
    o = synth.fill_host(synth.Spec(seed=0, stream=3, dist=synth.STUDENT_T3, sigma=1e-3,
                                   outlier_rate=1e-3, outlier_value=100.0), 0, n, synth.OUT_F32)
    assert (np.abs(o) == 100.0).mean() == pytest.approx(1e-3, rel=0.15)


def test_synth_windows_are_consistent():
    s = synth.Spec(seed=9, stream=4, rank=2, step=3, dist=synth.STUDENT_T3, sigma=1e-3)
    whole = synth.fill_host(s, 0, 5000, synth.OUT_BF16)
    assert (synth.fill_host(s, 1234, 77, synth.OUT_BF16) == whole[1234:1311]).all()


# ------------------------------------------------- gradient variants (not the method)


def test_fp32_gradients_match_torch_adam_demo_setting():
    """The page's runnable demo keeps fp32 gradients: 4 ranks, the demo MLP's
    19,210 parameters, lr 1e-2, 3 steps, against torch.optim.Adam on the average;
    the page's bar is max |diff| < 1e-5."""
    numel, world, lr = 19210, 4, 1e-2
    rng = np.random.default_rng(21)
    p = oracle.plan(numel, world)
    w0 = rng.normal(0, 0.05, numel).astype(np.float32)
    W = np.zeros(p["padded"], np.float32)
    W[:numel] = w0
    M, V = np.zeros_like(W), np.zeros_like(W)
    par = np.zeros(numel, np.uint16)
    ref = torch.nn.Parameter(torch.from_numpy(w0.copy()))
    opt = torch.optim.Adam([ref], lr=lr, betas=(B1, B2), eps=EPS, foreach=False, fused=False)
    for t in range(1, 4):
        rows = [rng.normal(0, 1e-2, numel).astype(np.float32) for _ in range(world)]
        grads = [np.pad(r, (0, p["padded"] - numel)) for r in rows]
        oracle.zero_step(numel, world, -1, grads, W, M, V, par, lr, B1, B2, EPS, t, grad_f32=True)
        acc = rows[0].copy()
        for r in rows[1:]:
            acc = acc + r
        ref.grad = torch.from_numpy(acc / np.float32(world))
        opt.step()
    st = opt.state[ref]
    w_ref = ref.detach().numpy()
    assert np.abs(W[:numel] - w_ref).max() < 1e-5
    assert np.allclose(W[:numel], w_ref, rtol=1e-6, atol=2e-8)
    m_ref = st["exp_avg"].numpy()
    assert np.allclose(M[:numel], m_ref, rtol=1e-6, atol=1e-6 * np.abs(m_ref).max())


def test_bf16_accumulation_rounds_each_partial_sum():
    """In bf16 (8 significant bits) 1 + 2^-8 ties to 1, twice; the fp32 sum is 1 + 2^-7.
    With beta1 = 0 the first moment is the averaged gradient itself."""
    h = 2.0**-8
    rows = [_bf16([1.0]), _bf16([h]), _bf16([h])]
    numel, world = 1, 3
    p = oracle.plan(numel, world)
    grads = [np.pad(r, (0, p["padded"] - numel)) for r in rows]

    def run(acc_bf16):
        W = np.zeros(p["padded"], np.float32)
        M, V = np.zeros_like(W), np.zeros_like(W)
        oracle.zero_step(numel, world, -1, grads, W, M, V, np.zeros(1, np.uint16), LR, 0.0, 0.0,
                         EPS, 1, acc_bf16=acc_bf16)
        return M[0]

    assert run(True) == np.float32(1.0) / np.float32(3.0)
    assert run(False) == np.float32(1.0 + 2.0**-7) / np.float32(3.0)
    # one rank: nothing is added, so the variant is the method (bf16 gradients)
    rng = np.random.default_rng(22)
    g = _bf16(rng.normal(0, 1e-3, 999))
    outs = []
    for acc in (False, True):
        W = rng.normal(0, 0.02, 999).astype(np.float32) * 0 + 0.01
        M, V, par = np.zeros(999, np.float32), np.zeros(999, np.float32), np.zeros(999, np.uint16)
        oracle.zero_step(999, 1, -1, [g], W, M, V, par, LR, B1, B2, EPS, 1, acc_bf16=acc)
        outs.append((W.copy(), M.copy()))
    assert (outs[0][0].view(np.uint32) == outs[1][0].view(np.uint32)).all()


def test_unit_gather_rows_brute_force():
    """FSDP2-style dim-0 sharding: numpy builds each rank's row blocks (ceil-sized
    chunks, zero rows past the end) and the gather must restore the tensors."""
    rng = np.random.default_rng(23)
    for _ in range(200):
        world = int(rng.integers(1, 9))
        shapes = [(int(rng.integers(1, 20)), int(rng.integers(1, 7)))
                  for _ in range(int(rng.integers(1, 5)))]
        tensors = [rng.integers(0, 2**16, r * c, dtype=np.uint64).astype(np.uint16).reshape(r, c)
                   for r, c in shapes]
        shards = []
        for k in range(world):
            parts = []
            for t in tensors:
                R = -(-t.shape[0] // world)
                block = np.zeros((R, t.shape[1]), np.uint16)
                rows = t[k * R:(k + 1) * R]
                block[:rows.shape[0]] = rows
                parts.append(block.ravel())
            shards.append(np.concatenate(parts))
        full = oracle.unit_gather_rows(shapes, world, shards)
        assert (full == np.concatenate([t.ravel() for t in tensors])).all(), (world, shapes)


def test_unit_gather_rows_one_tensor_with_divisible_rows_is_the_flat_gather():
    """One tensor whose rows divide by N: the row blocks are the flat shards."""
    rng = np.random.default_rng(24)
    rows, cols, world = 64, 10, 8
    shards = [rng.integers(0, 2**16, rows // world * cols, dtype=np.uint64).astype(np.uint16)
              for _ in range(world)]
    assert (oracle.unit_gather_rows([(rows, cols)], world, shards)
            == oracle.unit_gather(rows * cols, world, shards)).all()
