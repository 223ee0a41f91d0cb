// capi.cpp -- the extern "C" entry points of libzeroadam.so (include/zeroadam.h):
// argument checking, the shard planner, the fp32 scalars, kernel dispatch.
// Every entry point that launches work, or waits for it, opens an NVTX range
// named after itself for its whole duration (a no-op unless a profiler or
// another NVTX tool is attached).
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "zeroadam.h"
#include "internal.h"

namespace zeroadam {

int device_sm_count(int* sms) {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  if (dev < 64) {
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] > 0) {
      *sms = cache[dev];
      return 0;
    }
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    return -1;
  if (dev < 64) {
    std::lock_guard<std::mutex> lock(mu);
    cache[dev] = n;
  }
  *sms = n;
  return 0;
}

namespace {

// Scoped NVTX range.
struct Trace {
  explicit Trace(const char* name) { nvtxRangePushA(name); }
  ~Trace() { nvtxRangePop(); }
  Trace(const Trace&) = delete;
  Trace& operator=(const Trace&) = delete;
};

// zero_test_withhold_copies: read by every step launch (relaxed; a test sets it
// between launches).
std::atomic<int> g_withhold{0};

thread_local cudaError_t t_last_cuda = cudaSuccess;
thread_local std::string t_msg;

// ZERO_E_DEVICE, keeping the CUDA error for zero_strerror.
int device_error(cudaError_t e) {
  t_last_cuda = e == cudaSuccess ? cudaErrorNoDevice : e;
  return ZERO_E_DEVICE;
}

int launch_status(cudaError_t e) {
  if (e == cudaSuccess) return ZERO_OK;
  t_last_cuda = e;
  return e == cudaErrorNoDevice ? ZERO_E_DEVICE : ZERO_E_LAUNCH;
}

// Shard layout: ceil(numel/world) elements per rank, zero pad at the end
// ("Implementing ZeRO's Adam from scratch": shard size and _flatten).
int make_plan(int64_t numel, int32_t world, zero_plan_t* p) {
  if (world < 1 || world > ZERO_MAX_WORLD) return ZERO_E_WORLD;
  if (numel < 1) return ZERO_E_NUMEL;
  const int64_t shard = numel / world + (numel % world != 0 ? 1 : 0);
  if (shard > INT64_MAX / world) return ZERO_E_NUMEL;
  const int64_t padded = shard * world;
  // the byte counts below (at most 16 * numel) must not overflow
  if (numel > INT64_MAX / 16) return ZERO_E_NUMEL;
  p->numel = numel;
  p->world = world;
  p->shard = shard;
  p->padded = padded;
  p->pad = padded - numel;
  const uint64_t P = static_cast<uint64_t>(numel), S = static_cast<uint64_t>(shard);
  // "The three stages": bf16 param (2) + bf16 grad (2) + fp32 master/m/v (12)
  // per parameter; ZeRO-1 shards the 12, ZeRO-2 also the grad, ZeRO-3 all 16.
  p->bytes_dp = 16 * P;
  p->bytes_z1 = 4 * P + 12 * S;
  p->bytes_z2 = 2 * P + 14 * S;
  p->bytes_z3 = 16 * S;
  const double Pd = static_cast<double>(numel), Nd = static_cast<double>(world);
  p->formula_dp = 16.0 * Pd;
  p->formula_z1 = 4.0 * Pd + 12.0 * Pd / Nd;
  p->formula_z2 = 2.0 * Pd + 14.0 * Pd / Nd;
  p->formula_z3 = 16.0 * Pd / Nd;
  p->state_bytes_rank = 12 * S;
  // Ring collectives over the padded bf16 vector: reduce-scatter and
  // all-gather each send (N-1)/N of it per card.
  const double vec_bytes = 2.0 * static_cast<double>(padded);
  const double frac = (Nd - 1.0) / Nd;
  p->comm_dp = 2.0 * frac * vec_bytes;
  p->comm_z1 = p->comm_dp;
  p->comm_z2 = p->comm_dp;
  p->comm_z3 = 3.0 * frac * vec_bytes;
  return ZERO_OK;
}

int check_plan(const zero_plan_t* plan) {
  if (plan == nullptr) return ZERO_E_NULLPTR;
  if (plan->world < 1 || plan->world > ZERO_MAX_WORLD) return ZERO_E_WORLD;
  zero_plan_t ref;
  const int rc = make_plan(plan->numel, static_cast<int32_t>(plan->world), &ref);
  if (rc != ZERO_OK) return rc;
  if (ref.shard != plan->shard || ref.pad != plan->pad || ref.padded != plan->padded)
    return ZERO_E_PLAN;
  return ZERO_OK;
}

bool is_finite(double x) { return std::isfinite(x); }

struct Range {
  uintptr_t lo, hi;
};
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }
Range bytes_of(const void* p, int64_t first, int64_t count, int esize) {
  const uintptr_t b = reinterpret_cast<uintptr_t>(p) + static_cast<uintptr_t>(first) * esize;
  return {b, b + static_cast<uintptr_t>(count) * esize};
}
bool nonempty(Range r) { return r.hi > r.lo; }

// A step over [begin, end), checked: its launch and the byte ranges it
// touches (for the unit step's checks across its two parts).
struct PreparedStep {
  StepLaunch L;
  const void* g[ZERO_MAX_WORLD];  // gradient pointers at the range's first element
  Range outs[4];                  // master, m, v, param bytes written (L.n > 0)
  int gsize;                      // bytes per gradient element
  // gradient k's bytes read (L.n > 0)
  Range grad_bytes(int32_t k) const { return bytes_of(g[k], 0, L.n, gsize); }
};

// The checks of one step over [begin, end) (every step entry point).
int prepare_step(const zero_plan_t* plan, int32_t rank, int64_t begin, int64_t end,
                 const void* const* grad_ptrs, int32_t grad_layout, float* master, float* m,
                 float* v, void* param_bf16, int32_t param_layout, double lr, double beta1,
                 double beta2, double eps, int64_t t, void* stream, PreparedStep* ps) {
  int rc = check_plan(plan);
  if (rc != ZERO_OK) return rc;
  const int32_t N = static_cast<int32_t>(plan->world);
  if (rank != ZERO_ALL_RANKS && (rank < 0 || rank >= N)) return ZERO_E_RANK;
  const int32_t layout = grad_layout & ZERO_GRAD_LAYOUT_MASK;
  const int32_t gflags = grad_layout & ~ZERO_GRAD_LAYOUT_MASK;
  if (layout != ZERO_GRAD_FULL && layout != ZERO_GRAD_SHARD && layout != ZERO_GRAD_WINDOW)
    return ZERO_E_LAYOUT;
  if ((gflags & ~(ZERO_GRAD_F32 | ZERO_ACC_BF16)) != 0) return ZERO_E_LAYOUT;
  if (param_layout != ZERO_PARAM_FULL && param_layout != ZERO_PARAM_SHARD) return ZERO_E_LAYOUT;
  if (rank == ZERO_ALL_RANKS && (layout == ZERO_GRAD_SHARD || param_layout != ZERO_PARAM_FULL))
    return ZERO_E_LAYOUT;
  if (begin < 0 || end < begin) return ZERO_E_RANGE;
  if (!is_finite(lr) || !is_finite(eps) || !is_finite(beta1) || !is_finite(beta2) || lr < 0.0 ||
      eps < 0.0 || beta1 < 0.0 || beta1 >= 1.0 || beta2 < 0.0 || beta2 >= 1.0)
    return ZERO_E_HPARAM;
  if (t < 1) return ZERO_E_STEP;
  if (grad_ptrs == nullptr || master == nullptr || m == nullptr || v == nullptr ||
      param_bf16 == nullptr)
    return ZERO_E_NULLPTR;
  for (int32_t k = 0; k < N; ++k)
    if (grad_ptrs[k] == nullptr) return ZERO_E_NULLPTR;

  // The stepped range of global flat indices: the rank's (or every rank's)
  // real elements, intersected with [begin, end).
  int64_t lo = 0, hi = plan->numel;
  if (rank != ZERO_ALL_RANKS) {
    lo = static_cast<int64_t>(rank) * plan->shard;
    hi = lo + plan->shard;
    if (hi > plan->numel) hi = plan->numel;
  }
  const int64_t a = begin > lo ? begin : lo;
  const int64_t b = end < hi ? end : hi;
  const int64_t n = b > a ? b - a : 0;
  // Where each buffer holds global index a.
  const int64_t g_first = layout == ZERO_GRAD_FULL ? a : layout == ZERO_GRAD_SHARD ? a - lo
                                                                                   : a - begin;
  // master/m/v: all ranks' shards back to back (global index), or one
  // rank's shard (global index lo is its element 0).
  const int64_t s_first = rank == ZERO_ALL_RANKS ? a : a - lo;
  const int64_t p_first = param_layout == ZERO_PARAM_FULL ? a : a - lo;
  const int gsize = (gflags & ZERO_GRAD_F32) ? 4 : 2;

  auto misaligned = [](const void* p, uintptr_t k) {
    return (reinterpret_cast<uintptr_t>(p) & (k - 1)) != 0;
  };
  if (misaligned(master, 4) || misaligned(m, 4) || misaligned(v, 4) || misaligned(param_bf16, 2))
    return ZERO_E_ALIGN;
  for (int32_t k = 0; k < N; ++k)
    if (misaligned(grad_ptrs[k], gsize)) return ZERO_E_ALIGN;

  if (n > 0) {
    ps->outs[0] = bytes_of(master, s_first, n, 4);
    ps->outs[1] = bytes_of(m, s_first, n, 4);
    ps->outs[2] = bytes_of(v, s_first, n, 4);
    ps->outs[3] = bytes_of(param_bf16, p_first, n, 2);
    for (int i = 0; i < 4; ++i)
      for (int j = i + 1; j < 4; ++j)
        if (overlap(ps->outs[i], ps->outs[j])) return ZERO_E_ALIAS;
    for (int32_t k = 0; k < N; ++k) {
      const Range gk = bytes_of(grad_ptrs[k], g_first, n, gsize);
      for (int i = 0; i < 4; ++i)
        if (overlap(gk, ps->outs[i])) return ZERO_E_ALIAS;
    }
  }

  // Offset every pointer to the range's first element.
  for (int32_t k = 0; k < N; ++k)
    ps->g[k] = static_cast<const char*>(grad_ptrs[k]) + g_first * gsize;
  ps->gsize = gsize;

  StepLaunch& L = ps->L;
  L.grads = ps->g;
  L.world = N;
  L.grad_f32 = (gflags & ZERO_GRAD_F32) ? 1 : 0;
  L.acc_bf16 = (gflags & ZERO_ACC_BF16) ? 1 : 0;
  L.master = master + s_first;
  L.m = m + s_first;
  L.v = v + s_first;
  L.param = static_cast<uint16_t*>(param_bf16) + p_first;
  L.n = n;
  L.stream = static_cast<cudaStream_t>(stream);
  L.withhold = g_withhold.load(std::memory_order_relaxed);
  AdamScalars& sc = L.s;
  sc.b1 = static_cast<float>(beta1);
  sc.omb1 = static_cast<float>(1.0 - beta1);
  sc.b2 = static_cast<float>(beta2);
  sc.omb2 = static_cast<float>(1.0 - beta2);
  sc.bc1 = static_cast<float>(1.0 - std::pow(beta1, static_cast<double>(t)));
  sc.bc2 = static_cast<float>(1.0 - std::pow(beta2, static_cast<double>(t)));
  sc.lr = static_cast<float>(lr);
  sc.eps = static_cast<float>(eps);
  sc.world = static_cast<float>(N);
  sc.pow2_world = (N & (N - 1)) == 0 ? 1 : 0;
  sc.inv_world = static_cast<float>(1.0 / static_cast<double>(N));
  return ZERO_OK;
}

// A flat unit gather, checked: its launch and the byte ranges it touches.
struct PreparedGather {
  GatherLaunch L;
  Range out;  // the unit's bytes written
  // shard k's bytes read (empty for a shard that holds only padding)
  Range shard_bytes(int32_t k) const {
    int64_t cnt = L.numel - static_cast<int64_t>(k) * L.shard;
    if (cnt > L.shard) cnt = L.shard;
    if (cnt < 0) cnt = 0;
    return bytes_of(L.shards[k], 0, cnt, 2);
  }
};

int prepare_gather(const zero_plan_t* unit_plan, const void* const* shard_ptrs, void* full_bf16,
                   void* stream, PreparedGather* pg) {
  int rc = check_plan(unit_plan);
  if (rc != ZERO_OK) return rc;
  const int32_t N = static_cast<int32_t>(unit_plan->world);
  if (shard_ptrs == nullptr || full_bf16 == nullptr) return ZERO_E_NULLPTR;
  for (int32_t k = 0; k < N; ++k)
    if (shard_ptrs[k] == nullptr) return ZERO_E_NULLPTR;
  if (reinterpret_cast<uintptr_t>(full_bf16) & 1u) return ZERO_E_ALIGN;
  for (int32_t k = 0; k < N; ++k)
    if (reinterpret_cast<uintptr_t>(shard_ptrs[k]) & 1u) return ZERO_E_ALIGN;
  GatherLaunch& L = pg->L;
  L.shards = reinterpret_cast<const uint16_t* const*>(shard_ptrs);
  L.world = N;
  L.full = static_cast<uint16_t*>(full_bf16);
  L.numel = unit_plan->numel;
  L.shard = unit_plan->shard;
  L.stream = static_cast<cudaStream_t>(stream);
  L.withhold = g_withhold.load(std::memory_order_relaxed);
  pg->out = bytes_of(full_bf16, 0, unit_plan->numel, 2);
  for (int32_t k = 0; k < N; ++k) {
    const Range sk = pg->shard_bytes(k);
    if (nonempty(sk) && overlap(pg->out, sk)) return ZERO_E_ALIAS;
  }
  return ZERO_OK;
}

}  // namespace
}  // namespace zeroadam

using namespace zeroadam;

extern "C" {

int zero_plan(int64_t numel, int32_t world, zero_plan_t* out) {
  if (out == nullptr) return ZERO_E_NULLPTR;
  return make_plan(numel, world, out);
}

int zero_adam_step_range(const zero_plan_t* plan, int32_t rank, int64_t begin, int64_t end,
                         const void* const* grad_ptrs, int32_t grad_layout, float* master,
                         float* m, float* v, void* param_bf16, int32_t param_layout, double lr,
                         double beta1, double beta2, double eps, int64_t t, void* stream) {
  Trace trace("zero_adam_step_range");
  PreparedStep ps;
  const int rc = prepare_step(plan, rank, begin, end, grad_ptrs, grad_layout, master, m, v,
                              param_bf16, param_layout, lr, beta1, beta2, eps, t, stream, &ps);
  if (rc != ZERO_OK || ps.L.n == 0) return rc;
  return launch_status(launch_adam_step(ps.L));
}

int zero_adam_step(const zero_plan_t* plan, int32_t rank, const void* const* grad_ptrs,
                   int32_t grad_layout, float* master, float* m, float* v, void* param_bf16,
                   int32_t param_layout, double lr, double beta1, double beta2, double eps,
                   int64_t t, void* stream) {
  Trace trace("zero_adam_step");
  if ((grad_layout & ZERO_GRAD_LAYOUT_MASK) == ZERO_GRAD_WINDOW) return ZERO_E_LAYOUT;
  PreparedStep ps;
  const int rc = prepare_step(plan, rank, 0, INT64_MAX, grad_ptrs, grad_layout, master, m, v,
                              param_bf16, param_layout, lr, beta1, beta2, eps, t, stream, &ps);
  if (rc != ZERO_OK || ps.L.n == 0) return rc;
  return launch_status(launch_adam_step(ps.L));
}

int zero3_unit_step(const zero_plan_t* unit_plan, int32_t rank, const void* const* shard_ptrs,
                    void* full_bf16, const void* const* grad_ptrs, int32_t grad_layout,
                    float* master, float* m, float* v, void* param_bf16, int32_t param_layout,
                    double lr, double beta1, double beta2, double eps, int64_t t, void* stream) {
  Trace trace("zero3_unit_step");
  if ((grad_layout & ZERO_GRAD_LAYOUT_MASK) == ZERO_GRAD_WINDOW) return ZERO_E_LAYOUT;
  PreparedGather pg;
  int rc = prepare_gather(unit_plan, shard_ptrs, full_bf16, stream, &pg);
  if (rc != ZERO_OK) return rc;
  PreparedStep ps;
  rc = prepare_step(unit_plan, rank, 0, INT64_MAX, grad_ptrs, grad_layout, master, m, v,
                    param_bf16, param_layout, lr, beta1, beta2, eps, t, stream, &ps);
  if (rc != ZERO_OK) return rc;
  // The two parts run side by side: the gathered unit must not overlap what
  // the step reads or writes, and the shards must not overlap what it writes.
  if (ps.L.n > 0) {
    const int32_t N = static_cast<int32_t>(unit_plan->world);
    for (int i = 0; i < 4; ++i)
      if (overlap(pg.out, ps.outs[i])) return ZERO_E_ALIAS;
    for (int32_t k = 0; k < N; ++k) {
      const Range sk = pg.shard_bytes(k);
      for (int i = 0; i < 4; ++i)
        if (nonempty(sk) && overlap(sk, ps.outs[i])) return ZERO_E_ALIAS;
      if (overlap(pg.out, ps.grad_bytes(k))) return ZERO_E_ALIAS;
    }
  }
  return launch_status(launch_unit_step(pg.L, ps.L));
}

int zero_test_withhold_copies(int on) {
  const char* gate = std::getenv("ZEROADAM_TEST_HOOKS");
  if (gate == nullptr || std::strcmp(gate, "1") != 0) return ZERO_E_HOOK;
  return g_withhold.exchange(on != 0 ? 1 : 0);
}

int zero3_unit_gather(const zero_plan_t* unit_plan, const void* const* shard_ptrs,
                      void* full_bf16, void* stream) {
  Trace trace("zero3_unit_gather");
  PreparedGather pg;
  const int rc = prepare_gather(unit_plan, shard_ptrs, full_bf16, stream, &pg);
  if (rc != ZERO_OK) return rc;
  return launch_status(launch_unit_gather(pg.L));
}

int zero3_unit_gather_rows(int32_t ntensors, const int64_t* rows, const int64_t* cols,
                           int32_t world, const void* const* shard_ptrs, void* full_bf16,
                           void* stream) {
  Trace trace("zero3_unit_gather_rows");
  if (ntensors < 1 || ntensors > ZERO_MAX_UNIT_TENSORS) return ZERO_E_SHAPE;
  if (world < 1 || world > ZERO_MAX_WORLD) return ZERO_E_WORLD;
  if (rows == nullptr || cols == nullptr || shard_ptrs == nullptr || full_bf16 == nullptr)
    return ZERO_E_NULLPTR;
  int64_t per_rank[ZERO_MAX_UNIT_TENSORS], full_off[ZERO_MAX_UNIT_TENSORS],
      shard_off[ZERO_MAX_UNIT_TENSORS];
  int64_t total = 0, shard_len = 0;
  const int64_t lim = INT64_MAX / 4;
  for (int32_t i = 0; i < ntensors; ++i) {
    if (rows[i] < 1 || cols[i] < 1) return ZERO_E_SHAPE;
    if (rows[i] > lim / cols[i]) return ZERO_E_SHAPE;
    per_rank[i] = rows[i] / world + (rows[i] % world != 0 ? 1 : 0);
    full_off[i] = total;
    shard_off[i] = shard_len;
    total += rows[i] * cols[i];
    shard_len += per_rank[i] * cols[i];
    if (total > lim || shard_len > lim) return ZERO_E_SHAPE;
  }
  for (int32_t k = 0; k < world; ++k)
    if (shard_ptrs[k] == nullptr) return ZERO_E_NULLPTR;
  if (reinterpret_cast<uintptr_t>(full_bf16) & 1u) return ZERO_E_ALIGN;
  for (int32_t k = 0; k < world; ++k)
    if (reinterpret_cast<uintptr_t>(shard_ptrs[k]) & 1u) return ZERO_E_ALIGN;
  const Range out = bytes_of(full_bf16, 0, total, 2);
  for (int32_t k = 0; k < world; ++k)
    if (overlap(out, bytes_of(shard_ptrs[k], 0, shard_len, 2))) return ZERO_E_ALIAS;
  GatherRowsLaunch L;
  L.shards = reinterpret_cast<const uint16_t* const*>(shard_ptrs);
  L.world = world;
  L.ntensors = ntensors;
  L.rows = rows;
  L.cols = cols;
  L.rows_per_rank = per_rank;
  L.full_off = full_off;
  L.shard_off = shard_off;
  L.full = static_cast<uint16_t*>(full_bf16);
  L.stream = static_cast<cudaStream_t>(stream);
  L.withhold = g_withhold.load(std::memory_order_relaxed);
  return launch_status(launch_unit_gather_rows(L));
}

int zero_device_status(void) {
  Trace trace("zero_device_status");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return device_error(e);
  // Every kernel launched so far on this device, on any stream, has finished
  // (and set its word, if a wait gave up) before the words are taken.
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return device_error(e);
  static std::mutex mu;  // one caller at a time takes the words
  std::lock_guard<std::mutex> lock(mu);
  int step = 0, gather = 0;
  if (read_and_clear_step_status(&step) != 0) return device_error(cudaGetLastError());
  if (read_and_clear_gather_status(&gather) != 0) return device_error(cudaGetLastError());
  return step == 0 && gather == 0 ? ZERO_OK : ZERO_E_TIMEOUT;
}

const char* zero_strerror(int status) {
  switch (status) {
    case ZERO_OK: return "ok";
    case ZERO_E_NULLPTR: return "a required pointer is NULL";
    case ZERO_E_WORLD: return "world must be in [1, ZERO_MAX_WORLD]";
    case ZERO_E_NUMEL: return "numel must be >= 1 and world*shard must fit in int64";
    case ZERO_E_RANK: return "rank must be in [0, world) or ZERO_ALL_RANKS";
    case ZERO_E_STEP: return "t must be >= 1 (1-based step count)";
    case ZERO_E_ALIGN: return "bf16 pointers must be 2-byte and fp32 pointers 4-byte aligned";
    case ZERO_E_HPARAM: return "lr and eps must be finite and >= 0, betas in [0, 1)";
    case ZERO_E_LAYOUT: return "unknown layout, or a shard layout with ZERO_ALL_RANKS";
    case ZERO_E_PLAN: return "plan fields differ from zero_plan(numel, world)";
    case ZERO_E_ALIAS: return "an output buffer overlaps another buffer";
    case ZERO_E_DEVICE:
      t_msg = std::string("no usable CUDA device, or the device reported an error: ") +
              cudaGetErrorString(t_last_cuda == cudaSuccess ? cudaErrorNoDevice : t_last_cuda);
      return t_msg.c_str();
    case ZERO_E_RANGE: return "the window must satisfy 0 <= begin <= end";
    case ZERO_E_SHAPE: return "ntensors in [1, ZERO_MAX_UNIT_TENSORS] and sizes >= 1 required";
    case ZERO_E_TIMEOUT: return "a kernel gave up a bounded wait; that step's outputs are incomplete";
    case ZERO_E_HOOK: return "test hooks are off: they need ZEROADAM_TEST_HOOKS=1 in the environment";
    case ZERO_E_LAUNCH:
      t_msg = std::string("kernel launch failed: ") + cudaGetErrorString(t_last_cuda);
      return t_msg.c_str();
    default: return "unknown status";
  }
}

int zero_version(void) { return 0x000100; }

}  // extern "C"
