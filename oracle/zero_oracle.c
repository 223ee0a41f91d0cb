/*
 * zero_oracle.c -- the ORACLE: a plain, slow CPU statement of the ZeRO
 * stage-1/2 Adam step, the ZeRO-3 unit gather and the shard planner.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this.  It shares no code, header or
 * constant with the CUDA library; the two meet only in the seeded inputs.
 *
 * Source of the method: "ZeRO and FSDP: partitioning the optimizer states, the
 * gradients and the parameters" (AI infra handbooks), sections "The three
 * stages" (table), "Implementing ZeRO's Adam from scratch" (class ZeroAdam:
 * __init__, _flatten, step, state_bytes) and "Exercises".
 *
 * Precision.  The page keeps fp32 master weights and fp32 moments and bf16
 * parameters and gradients ("The three stages": mixed-precision Adam; the
 * ZeroAdam master-slice comment).  Every floating-point operation below is one
 * IEEE binary32 operation, rounded to nearest even, in the order the page's
 * tensor expressions evaluate them; compiled with -ffp-contract=off and
 * without fast-math, denormals kept.  The step's scalars (1-b1, 1-b1^t, ...)
 * are Python floats on the page, i.e. doubles, and meet the fp32 tensors
 * once: they are computed in double and rounded to binary32 once.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC -lm
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "zero_oracle.h"

/* ---------------------------------------------------------------- planner */

/*
 * ZeroAdam.__init__ and _flatten: numel = sum of parameter sizes, each rank
 * is responsible for shard = ceil(numel / world) elements, the flat vector has
 * shard*world elements with the tail zero-padded, and rank r holds
 * [r*shard, (r+1)*shard).
 *
 * Model states per card ("The three stages" table; "Exercises" answer):
 * mixed-precision Adam keeps, per parameter, a bf16 parameter (2 B), a bf16
 * gradient (2 B), and fp32 master, first and second moment (4 B each).  A
 * stage either replicates a component (Psi elements on every card) or
 * partitions it (shard elements per card):
 *   DP     : nothing partitioned
 *   ZeRO-1 : the optimizer states (master, m, v)
 *   ZeRO-2 : + the gradients
 *   ZeRO-3 : + the parameters
 * bytes_* are those sums with the padded shard; formula_* are the table's
 * expressions 16 Psi, 4 Psi + 12 Psi/N, 2 Psi + 14 Psi/N, 16 Psi/N evaluated
 * as real numbers.
 */
int oracle_plan(int64_t numel, int32_t world, oracle_plan_t* out) {
  if (out == NULL || numel < 1 || world < 1) return -1;
  int64_t shard = numel / world;
  if (shard * (int64_t)world < numel) shard += 1; /* ceil */
  if (shard > INT64_MAX / world) return -1;

  memset(out, 0, sizeof(*out));
  out->numel = numel;
  out->world = world;
  out->shard = shard;
  out->padded = shard * (int64_t)world;
  out->pad = out->padded - numel;

  /* component sizes in bytes per element and which stage partitions them */
  enum { PARAM, GRAD, MASTER, MOM1, MOM2, NCOMP };
  const uint64_t size[NCOMP] = {2, 2, 4, 4, 4};
  /* first stage (0=DP,1,2,3) at which the component is partitioned */
  const int part_from[NCOMP] = {3, 2, 1, 1, 1};
  uint64_t bytes[4];
  for (int stage = 0; stage < 4; ++stage) {
    uint64_t b = 0;
    for (int c = 0; c < NCOMP; ++c) {
      const int partitioned = (stage >= part_from[c]);
      const uint64_t count = partitioned ? (uint64_t)shard : (uint64_t)numel;
      b += size[c] * count;
    }
    bytes[stage] = b;
  }
  out->bytes_dp = bytes[0];
  out->bytes_z1 = bytes[1];
  out->bytes_z2 = bytes[2];
  out->bytes_z3 = bytes[3];

  const double P = (double)numel, N = (double)world;
  out->formula_dp = 16.0 * P;
  out->formula_z1 = 4.0 * P + 12.0 * P / N;
  out->formula_z2 = 2.0 * P + 14.0 * P / N;
  out->formula_z3 = 16.0 * P / N;
  /* ZeroAdam.state_bytes: master + m + v of this rank, fp32 */
  out->state_bytes_rank = 3u * 4u * (uint64_t)shard;

  /*
   * Bytes each card sends per step ("The three stages" table, last column;
   * "Exercises", second answer).  The collectives run on the padded bf16
   * vector (2 bytes x padded).  In a ring, a reduce-scatter and an all-gather
   * each send (N-1)/N of the vector per card, and an all-reduce is one of
   * each.  DP all-reduces the gradients; ZeRO-1 and ZeRO-2 reduce-scatter the
   * gradients and all-gather the parameters; ZeRO-3 all-gathers the
   * parameters in the forward and again in the backward pass and
   * reduce-scatters the gradients.
   */
  const double vec = 2.0 * (double)out->padded;
  const double ring_share = ((double)world - 1.0) / (double)world;
  const double reduce_scatter = ring_share * vec;
  const double all_gather = ring_share * vec;
  out->comm_dp = reduce_scatter + all_gather;
  out->comm_z1 = reduce_scatter + all_gather;
  out->comm_z2 = reduce_scatter + all_gather;
  out->comm_z3 = all_gather + all_gather + reduce_scatter;
  return 0;
}

/* ------------------------------------------------------------- bf16 <-> f32 */

/* A bf16 value is the upper half of a binary32: widening is exact. */
float oracle_bf16_to_f32(uint16_t h) {
  const uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/*
 * Round a binary32 to the nearest bf16, ties to the candidate whose last bit
 * is zero (IEEE round-to-nearest-even).  The two candidates are the value cut
 * to 16 bits (toward zero in magnitude) and the next bf16 up in magnitude; the
 * 16 dropped bits say which is nearer.  NaN stays NaN (quiet bit set).
 */
uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
  const uint32_t toward_zero = u >> 16;
  const uint32_t away = toward_zero + 1u; /* may carry into the exponent: correct */
  const uint32_t dropped = u & 0xffffu;
  if (dropped < 0x8000u) return (uint16_t)toward_zero;
  if (dropped > 0x8000u) return (uint16_t)away;
  return (uint16_t)((toward_zero & 1u) ? away : toward_zero);
}

/* ---------------------------------------------------------------- scalars */

/*
 * ZeroAdam.step: t is incremented before use (self.t += 1), so the t given
 * here is already the 1-based step number.  The Python-float expressions
 * 1 - b1, 1 - b2, 1 - b1**t, 1 - b2**t are computed in double and each is
 * rounded to binary32 when it meets an fp32 tensor.
 */
void oracle_scalars(double lr, double beta1, double beta2, double eps, int64_t t, int32_t world,
                    oracle_scalars_t* s) {
  s->b1 = (float)beta1;
  s->omb1 = (float)(1.0 - beta1);
  s->b2 = (float)beta2;
  s->omb2 = (float)(1.0 - beta2);
  s->bc1 = (float)(1.0 - pow(beta1, (double)t));
  s->bc2 = (float)(1.0 - pow(beta2, (double)t));
  s->lr = (float)lr;
  s->eps = (float)eps;
  s->world = (float)world;
}

/* ------------------------------------------------------------ one element */

/* Rank k's gradient at buffer index idx, widened to fp32 (exact). */
static float oracle_grad(const void* const* grads, int grad_f32, int32_t k, int64_t idx) {
  if (grad_f32) return ((const float*)grads[k])[idx];
  return oracle_bf16_to_f32(((const uint16_t*)grads[k])[idx]);
}

/*
 * reduce_scatter_tensor of one element: the ranks' gradients summed in rank
 * order 0..N-1 in fp32, starting from rank 0's value.  Variant (not the
 * method): acc_bf16 rounds every partial sum to bf16, what a reduce-scatter
 * on bf16 buffers delivers.
 */
static float oracle_reduce(const void* const* grads, int grad_f32, int acc_bf16, int32_t world,
                           int64_t idx) {
  float acc = oracle_grad(grads, grad_f32, 0, idx);
  if (acc_bf16) acc = oracle_bf16_to_f32(oracle_f32_to_bf16(acc));
  for (int32_t k = 1; k < world; ++k) {
    acc = acc + oracle_grad(grads, grad_f32, k, idx);
    if (acc_bf16) acc = oracle_bf16_to_f32(oracle_f32_to_bf16(acc));
  }
  return acc;
}

/*
 * One flat element of ZeroAdam.step, in the page's order, from the summed
 * gradient acc:
 *   g /= world                g  = g / N
 *   m.mul_(b1).add_(g, alpha=1-b1)           m = m*b1 + (1-b1)*g
 *   v.mul_(b2).addcmul_(g, g, value=1-b2)    v = v*b2 + ((1-b2)*g)*g
 *   m_hat = m / (1 - b1**t);  v_hat = v / (1 - b2**t)
 *   master -= lr * m_hat / (v_hat.sqrt() + eps)
 *                                            w = w - (lr*m_hat) / (sqrt(v_hat)+eps)
 *   all_gather + copy into p.data            p = bf16(w)  (bf16 parameters)
 */
static void oracle_adam_element(float acc, const oracle_scalars_t* s, float* w, float* m,
                                float* v, uint16_t* p) {
  const float g = acc / s->world;

  float mm = *m, vv = *v, ww = *w;
  mm = mm * s->b1;
  mm = mm + s->omb1 * g;
  vv = vv * s->b2;
  vv = vv + (s->omb2 * g) * g;
  const float m_hat = mm / s->bc1;
  const float v_hat = vv / s->bc2;
  const float denom = sqrtf(v_hat) + s->eps;
  const float upd = (s->lr * m_hat) / denom;
  ww = ww - upd;

  *m = mm;
  *v = vv;
  *w = ww;
  *p = oracle_f32_to_bf16(ww);
}

/* ---------------------------------------------------------------- the step */

/*
 * ZeroAdam.step for rank `rank` (or every rank in turn when rank < 0), over
 * the global flat indices [i0, i1) only (pass 0, padded for the whole vector).
 *
 * Every array is addressed by global flat index minus its own base:
 *   grads[k][i - grad_base]    rank k's bf16 gradient (bits)
 *   master/m/v[i - state_base] fp32 state (state_base = 0 when the array holds
 *                              all ranks' shards back to back, r*shard when it
 *                              holds rank r's shard only)
 *   param[i - param_base]      bf16 parameters (bits)
 * Indices >= numel are the zero padding: their gradient is zero, so their
 * update is exactly zero and their state stays zero; _flatten's tail is
 * dropped when the gathered vector is copied back into the parameters.  The
 * oracle therefore neither reads nor writes any index >= numel.
 */
int oracle_zero_step_ex(const oracle_plan_t* plan, int32_t rank, int64_t i0, int64_t i1,
                        const void* const* grads, int64_t grad_base, int grad_f32, int acc_bf16,
                        float* master, float* m, float* v, int64_t state_base, uint16_t* param,
                        int64_t param_base, double lr, double beta1, double beta2, double eps,
                        int64_t t) {
  if (plan == NULL || grads == NULL || master == NULL || m == NULL || v == NULL || param == NULL)
    return -1;
  if (t < 1 || rank >= plan->world || plan->world > ORACLE_MAX_WORLD) return -1;
  oracle_scalars_t s;
  oracle_scalars(lr, beta1, beta2, eps, t, (int32_t)plan->world, &s);

  const int32_t r_first = rank < 0 ? 0 : rank;
  const int32_t r_last = rank < 0 ? (int32_t)plan->world - 1 : rank;
  for (int32_t r = r_first; r <= r_last; ++r) {
    int64_t lo = (int64_t)r * plan->shard;
    int64_t hi = lo + plan->shard;
    if (hi > plan->numel) hi = plan->numel;
    if (lo < i0) lo = i0;
    if (hi > i1) hi = i1;
    for (int64_t i = lo; i < hi; ++i) {
      const float acc =
          oracle_reduce(grads, grad_f32, acc_bf16, (int32_t)plan->world, i - grad_base);
      oracle_adam_element(acc, &s, &master[i - state_base], &m[i - state_base],
                          &v[i - state_base], &param[i - param_base]);
    }
  }
  return 0;
}

/* The method: bf16 gradients, fp32 rank-ordered sum. */
int oracle_zero_step(const oracle_plan_t* plan, int32_t rank, int64_t i0, int64_t i1,
                     const uint16_t* const* grads, int64_t grad_base, float* master, float* m,
                     float* v, int64_t state_base, uint16_t* param, int64_t param_base, double lr,
                     double beta1, double beta2, double eps, int64_t t) {
  return oracle_zero_step_ex(plan, rank, i0, i1, (const void* const*)grads, grad_base, 0, 0,
                             master, m, v, state_base, param, param_base, lr, beta1, beta2, eps,
                             t);
}

/*
 * Plain data parallelism, for the invariant "sharding changes nothing": every
 * card all-reduces (sums in rank order, then averages) the full gradient, then
 * runs the same Adam on the full, unpartitioned fp32 vectors and writes every
 * bf16 parameter.  Two passes, as DP does them: average, then update.
 */
int oracle_dp_step(int64_t numel, int32_t world, const uint16_t* const* grads, float* master,
                   float* m, float* v, uint16_t* param, double lr, double beta1, double beta2,
                   double eps, int64_t t) {
  if (numel < 0 || world < 1 || t < 1 || grads == NULL) return -1;
  oracle_scalars_t s;
  oracle_scalars(lr, beta1, beta2, eps, t, world, &s);
  float* avg = (float*)malloc((size_t)(numel > 0 ? numel : 1) * sizeof(float));
  if (avg == NULL) return -2;
  for (int64_t i = 0; i < numel; ++i) {
    float acc = oracle_bf16_to_f32(grads[0][i]);
    for (int32_t k = 1; k < world; ++k) acc = acc + oracle_bf16_to_f32(grads[k][i]);
    avg[i] = acc / s.world;
  }
  for (int64_t i = 0; i < numel; ++i) {
    const float g = avg[i];
    float mm = m[i] * s.b1;
    mm = mm + s.omb1 * g;
    float vv = v[i] * s.b2;
    vv = vv + (s.omb2 * g) * g;
    const float m_hat = mm / s.bc1;
    const float v_hat = vv / s.bc2;
    const float upd = (s.lr * m_hat) / (sqrtf(v_hat) + s.eps);
    m[i] = mm;
    v[i] = vv;
    master[i] = master[i] - upd;
    param[i] = oracle_f32_to_bf16(master[i]);
  }
  free(avg);
  return 0;
}

/* ----------------------------------------------------------- ZeRO-3 gather */

/*
 * ZeRO-3 unit all-gather ("ZeRO-3 and FSDP": before a unit is used, all-gather
 * its complete parameters): rank r's shard of shard = ceil(U/N) elements lands
 * at [r*shard, (r+1)*shard) of the unit, and the padded tail beyond U is
 * dropped.
 */
int oracle_unit_gather(int64_t unit_numel, int32_t world, const uint16_t* const* shards,
                       uint16_t* full) {
  oracle_plan_t p;
  if (oracle_plan(unit_numel, world, &p) != 0 || shards == NULL || full == NULL) return -1;
  for (int32_t r = 0; r < world; ++r)
    for (int64_t j = 0; j < p.shard; ++j) {
      const int64_t idx = (int64_t)r * p.shard + j;
      if (idx < unit_numel) full[idx] = shards[r][j];
    }
  return 0;
}

/* oracle_f32_to_bf16 over an array (for the tests' convenience). */
void oracle_f32_to_bf16_array(const float* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16(x[i]);
}

/*
 * FSDP2-style unit gather ("ZeRO-3 and FSDP": FSDP2 keeps every parameter as a
 * DTensor sharded along dimension 0; each rank holds a block of rows).  The
 * unit is ntensors row-major tensors, tensor i of rows[i] x cols[i].  With
 * R = ceil(rows[i] / world) rows per rank, rank r holds rows
 * [r*R, min((r+1)*R, rows[i])) of tensor i, stored as R x cols[i] elements
 * (rows past the tensor's end are padding); its shard is those blocks for
 * i = 0, 1, ... back to back.  The gathered unit is the tensors back to back.
 * Element (i, row, col) of the unit comes from rank row / R, local row
 * row - rank*R.
 */
int oracle_unit_gather_rows(int32_t ntensors, const int64_t* rows, const int64_t* cols,
                            int32_t world, const uint16_t* const* shards, uint16_t* full) {
  if (ntensors < 1 || world < 1 || rows == NULL || cols == NULL || shards == NULL || full == NULL)
    return -1;
  int64_t full_off = 0, shard_off = 0;
  for (int32_t i = 0; i < ntensors; ++i) {
    if (rows[i] < 1 || cols[i] < 1) return -1;
    int64_t R = rows[i] / world;
    if (R * world < rows[i]) R += 1;
    for (int64_t row = 0; row < rows[i]; ++row) {
      const int64_t r = row / R;
      const int64_t local = row - r * R;
      for (int64_t col = 0; col < cols[i]; ++col)
        full[full_off + row * cols[i] + col] = shards[r][shard_off + local * cols[i] + col];
    }
    full_off += rows[i] * cols[i];
    shard_off += R * cols[i];
  }
  return 0;
}
