"""The pins bite: each plausible mistake planted in a copy of the oracle fails them.

A mutant is the oracle's C source with one textual change, compiled on the CPU
into a temporary library; the pin suite then runs against it in a subprocess
(ZERO_ORACLE_SO) and must fail.  Nothing here touches a GPU.
"""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "zero_oracle.c")

MUTANTS = {
    "beta1_to_beta2_in_m": ("mm = mm * s->b1;", "mm = mm * s->b2;"),
    "eps_inside_sqrt": ("sqrtf(v_hat) + s->eps", "sqrtf(v_hat + s->eps)"),
    "no_average": ("const float g = acc / s->world;", "const float g = acc;"),
    "reverse_rank_order": (
        "float acc = oracle_grad(grads, grad_f32, 0, idx);\n"
        "  if (acc_bf16) acc = oracle_bf16_to_f32(oracle_f32_to_bf16(acc));\n"
        "  for (int32_t k = 1; k < world; ++k) {",
        "float acc = oracle_grad(grads, grad_f32, world - 1, idx);\n"
        "  if (acc_bf16) acc = oracle_bf16_to_f32(oracle_f32_to_bf16(acc));\n"
        "  for (int32_t k = world - 2; k >= 0; --k) {"),
    "bf16_sum_not_rounded": (
        "    acc = acc + oracle_grad(grads, grad_f32, k, idx);\n"
        "    if (acc_bf16) acc = oracle_bf16_to_f32(oracle_f32_to_bf16(acc));",
        "    acc = acc + oracle_grad(grads, grad_f32, k, idx);"),
    "f32_grads_truncated": ("if (grad_f32) return ((const float*)grads[k])[idx];",
                            "if (grad_f32) return oracle_bf16_to_f32("
                            "(uint16_t)(*(const uint32_t*)&((const float*)grads[k])[idx] >> 16));"),
    "no_bias_correction_m": ("const float m_hat = mm / s->bc1;", "const float m_hat = mm;"),
    "bias_power_t_minus_1": ("pow(beta2, (double)t)", "pow(beta2, (double)(t - 1))"),
    "update_sign": ("ww = ww - upd;", "ww = ww + upd;"),
    "v_missing_g_factor": ("vv = vv + (s->omb2 * g) * g;", "vv = vv + (s->omb2 * g);"),
    "scalar_in_single": ("s->omb1 = (float)(1.0 - beta1);", "s->omb1 = 1.0f - (float)beta1;"),
    "bf16_truncate": ("if (dropped < 0x8000u) return (uint16_t)toward_zero;",
                      "if (dropped < 0xffffu) return (uint16_t)toward_zero;"),
    "bf16_ties_away": ("return (uint16_t)((toward_zero & 1u) ? away : toward_zero);",
                       "return (uint16_t)away;"),
    "shard_floor": ("if (shard * (int64_t)world < numel) shard += 1; /* ceil */", ""),
    "grad_not_partitioned_in_z2": ("const int part_from[NCOMP] = {3, 2, 1, 1, 1};",
                                   "const int part_from[NCOMP] = {3, 3, 1, 1, 1};"),
    "gather_wrong_shard": ("if (idx < unit_numel) full[idx] = shards[r][j];",
                           "if (idx < unit_numel) full[idx] = shards[(r + 1) % world][j];"),
    "dp_step_no_average": ("avg[i] = acc / s.world;", "avg[i] = acc;"),
    "rows_shard_offset_unpadded": ("    shard_off += R * cols[i];",
                                   "    shard_off += (rows[i] / world) * cols[i];"),
    "rows_local_row_from_next_rank": ("      const int64_t local = row - r * R;",
                                      "      const int64_t local = row - r * R + (r > 0 ? 1 : 0);"),
    "no_bias_correction_v": ("const float v_hat = vv / s->bc2;", "const float v_hat = vv;"),
    "param_from_old_master": ("  ww = ww - upd;\n\n  *m = mm;\n  *v = vv;\n  *w = ww;\n  *p = oracle_f32_to_bf16(ww);",
                              "  *p = oracle_f32_to_bf16(ww);\n  ww = ww - upd;\n\n  *m = mm;\n  *v = vv;\n  *w = ww;"),
    "zero3_one_gather": ("out->comm_z3 = all_gather + all_gather + reduce_scatter;",
                         "out->comm_z3 = all_gather + reduce_scatter;"),
    "ring_share_whole_vector": ("const double ring_share = ((double)world - 1.0) / (double)world;",
                                "const double ring_share = 1.0;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_fails_the_pins(name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    with tempfile.TemporaryDirectory() as td:
        c = os.path.join(td, "zero_oracle.c")
        with open(c, "w") as f:
            f.write(src.replace(old, new))
        for h in ("zero_oracle.h",):
            with open(os.path.join(ROOT, "oracle", h)) as fi, open(os.path.join(td, h), "w") as fo:
                fo.write(fi.read())
        so = os.path.join(td, "libmutant.so")
        subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                        "-shared", "-o", so, c, "-lm"], check=True)
        env = dict(os.environ, ZERO_ORACLE_SO=so)
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                            os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
