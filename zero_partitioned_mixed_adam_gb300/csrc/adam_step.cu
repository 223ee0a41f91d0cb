// adam_step.cu -- the fused ZeRO-1/2 optimizer step on sm_103a.
//
// One pass over the stepped flat range does all of "ZeRO and FSDP" ->
// "Implementing ZeRO's Adam from scratch", ZeroAdam.step:
//   reduce-scatter + average  : sum of the N ranks' gradients, fp32, in rank
//                               order 0..N-1, divided by N
//   Adam + bias correction    : fp32 master, m, v updated in place
//   all-gather + unflatten    : bf16 (round to nearest even) of the new master
//                               stored straight into the flat parameter buffer
// The reduced gradient never leaves registers.  Per element the kernel moves
// N*sizeof(grad) (gradients) + 12 (state read) + 12 (state write) + 2 (bf16
// parameter) bytes and does ~20 fp32 operations: it is bound by HBM
// bandwidth, so it is written as a streaming kernel (16-byte vector
// loads/stores, a persistent grid-stride loop of 512-thread blocks sized to
// the SM count) and uses no tensor cores.  At N >= 5 with aligned buffers a
// TMA-staged variant replaces it: the gradients are bulk-copied in rank groups
// into a shared-memory ring, one CTA per SM.
//
// Bit-exactness: every operation is an explicit round-to-nearest intrinsic
// (__fadd_rn, __fmul_rn, __fdiv_rn, __fsqrt_rn), so nvcc cannot contract any
// pair into an FMA; the library is built without fast-math, so denormals are
// kept and division and square root are IEEE-correct.  The one rewrite is
// g/N -> g*(1/N) when N is a power of two, which is the same correctly
// rounded real number (1/N is exact).
//
// Variants (template parameters): gradients in bf16 (the mixed-precision
// setting) or fp32 (the page's runnable demo keeps fp32 gradients); the sum
// over ranks kept in fp32 (the method) or rounded to bf16 after every
// addition (what a reduce-scatter on bf16 buffers delivers).
#include <cuda_bf16.h>

#include <mutex>
#include <unordered_map>

#include "gather_ring.h"
#include "internal.h"
#include "tma_ops.h"

namespace zeroadam {
namespace {

constexpr int kThreads = 512;
constexpr int kTableRuntime = 1024;  // gradient-pointer table of the any-N kernel
// 1 when the register-staged kernel's instance has a fixed power-of-two N.
template <int NT>
constexpr int kPow2 = (NT > 0 && (NT & (NT - 1)) == 0) ? 1 : 0;

// Loads.  The gradients are never written while the kernel runs, so they may
// take the read-only (non-coherent) path.  master/m/v are read and then
// overwritten in place, so they take the coherent path with an evict-first
// hint: nothing is read twice.
template <typename T>
__device__ __forceinline__ T ld_grad(const T* p) {
  return __ldg(p);
}
template <typename T>
__device__ __forceinline__ T ld_state(const T* p) {
  return __ldcs(p);
}

template <int CAP>
struct StepArgs {
  const void* g[CAP];  // rank k's gradient, at the range's first element
  float* master;
  float* m;
  float* v;
  uint16_t* param;
  int64_t n;     // elements in the range
  int64_t nvec;  // 8-element vectors in the body [head, head + 8*nvec)
  int32_t head;  // scalar elements before the body
  int32_t world;
  int32_t gvec, svec, pvec;  // gradients / state / parameters 16-byte aligned in the body
  AdamScalars s;
};

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  return static_cast<uint32_t>(f32_to_bf16_rn(lo)) |
         (static_cast<uint32_t>(f32_to_bf16_rn(hi)) << 16);
}

// acc[j] += element j of one 16-byte vector of 8 bf16 (fp32 sum).
__device__ __forceinline__ void accumulate_bf16x8(float acc[8], const uint4 r) {
  acc[0] = __fadd_rn(acc[0], bf16_lo(r.x));
  acc[1] = __fadd_rn(acc[1], bf16_hi(r.x));
  acc[2] = __fadd_rn(acc[2], bf16_lo(r.y));
  acc[3] = __fadd_rn(acc[3], bf16_hi(r.y));
  acc[4] = __fadd_rn(acc[4], bf16_lo(r.z));
  acc[5] = __fadd_rn(acc[5], bf16_hi(r.z));
  acc[6] = __fadd_rn(acc[6], bf16_lo(r.w));
  acc[7] = __fadd_rn(acc[7], bf16_hi(r.w));
}

// One step of the running sum over ranks.
template <bool ABF16>
__device__ __forceinline__ float acc_add(float acc, float x) {
  const float s = __fadd_rn(acc, x);
  if (ABF16) return bf16_to_f32(f32_to_bf16_rn(s));
  return s;
}

// Adam with bias correction on one element, in ZeroAdam.step's order.
//
// A zero numerator skips its division: for x > 0, (+-0) / x is exactly +-0,
// the value the IEEE division returns.  That includes the average over ranks
// when N is not a power of two (a sum of exactly zero gradients divided by N:
// at N = 5..7 with a tenth of the sums zero, the division's slow path took the
// staged kernel from 0.96-1.02 to 0.79-0.85 of the copy peak on GB300).
// bc1 = 1 - b1^t and bc2 = 1 - b2^t are > 0 (beta in [0, 1), t >= 1); the
// last division is skipped only when its denominator is > 0 (0 / 0 still goes
// through the division and gives NaN).
// Elements whose gradient is exactly zero every step (untouched rows, dead
// units; the GPT-2 workload's 10 % mask) keep m = v = 0, and without the
// shortcut their divisions take the slow path of the IEEE division sequence.
// POW2 = 1: N is a power of two, known when the kernel is compiled (the
// register-staged kernel's fixed-N instances), so the average is always the
// exact multiplication by 1/N and no division code is generated; POW2 = 0:
// decided at run time from s.pow2_world.
template <int POW2>
__device__ __forceinline__ void adam_element(float gsum, const AdamScalars& s, float& w, float& m,
                                             float& v) {
  float g;
  if (POW2 || s.pow2_world)
    g = __fmul_rn(gsum, s.inv_world);
  else
    g = gsum == 0.0f ? gsum : __fdiv_rn(gsum, s.world);
  m = __fadd_rn(__fmul_rn(m, s.b1), __fmul_rn(s.omb1, g));
  v = __fadd_rn(__fmul_rn(v, s.b2), __fmul_rn(__fmul_rn(s.omb2, g), g));
  const float m_hat = (m == 0.0f) ? m : __fdiv_rn(m, s.bc1);
  const float v_hat = (v == 0.0f) ? v : __fdiv_rn(v, s.bc2);
  const float denom = __fadd_rn(__fsqrt_rn(v_hat), s.eps);
  const float num = __fmul_rn(s.lr, m_hat);
  w = __fsub_rn(w, (num == 0.0f && denom > 0.0f) ? num : __fdiv_rn(num, denom));
}

// The same update with the zero-numerator shortcut taken without a branch:
// every lane runs the divisions and the square root on normal operands (1.0
// stands in for a zero numerator, and 1/1 for the last division's shortcut
// case; the square root of v_hat = +-0 is +-0, taken from v_hat), then selects
// the shortcut's result.  With a tenth of the gradients exactly zero the
// square root of 0 had cost 1 % at N = 8 and 6 % at N = 5 on GB300; in the
// register-staged kernel's branching form the same guard was slower.  The
// values are those of adam_element bit for bit.  The staged kernels use this
// form: with some exact-zero gradients (the GPT-2 workload's 10 % mask) the
// branching form diverges within warps, and the staged kernels' best consumer
// count then moved with the fraction of zeros (measured on GB300 at N = 8: 24
// warps 1.00-1.05 of the copy peak depending on the data, this form 1.03-1.05
// at 22 warps).
__device__ __forceinline__ void adam_element_uniform(float gsum, const AdamScalars& s, float& w,
                                                     float& m, float& v) {
  float g;
  if (s.pow2_world) {  // the same for every thread of the launch
    g = __fmul_rn(gsum, s.inv_world);
  } else {
    const bool gz = gsum == 0.0f;
    const float gq = __fdiv_rn(gz ? 1.0f : gsum, s.world);
    g = gz ? gsum : gq;
  }
  m = __fadd_rn(__fmul_rn(m, s.b1), __fmul_rn(s.omb1, g));
  v = __fadd_rn(__fmul_rn(v, s.b2), __fmul_rn(__fmul_rn(s.omb2, g), g));
  const bool mz = m == 0.0f, vz = v == 0.0f;
  const float mq = __fdiv_rn(mz ? 1.0f : m, s.bc1);
  const float vq = __fdiv_rn(vz ? 1.0f : v, s.bc2);
  const float m_hat = mz ? m : mq;
  const float v_hat = vz ? v : vq;
  const float rt = __fsqrt_rn(vq);  // a normal operand: 1 / bc2 when v == 0
  const float denom = __fadd_rn(vz ? v_hat : rt, s.eps);  // sqrt(+-0) = +-0
  const float num = __fmul_rn(s.lr, m_hat);
  const bool z = num == 0.0f && denom > 0.0f;
  const float q = __fdiv_rn(z ? 1.0f : num, z ? 1.0f : denom);
  w = __fsub_rn(w, z ? num : q);
}

// 8 gradients of one rank as fp32, loaded as 16-byte vectors.
template <bool GF32>
struct GradVec;

template <>
struct GradVec<false> {  // 8 bf16 = one 16-byte vector
  uint4 r;
  __device__ __forceinline__ void load(const void* p, int64_t e0) {
    r = ld_grad(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p) + e0));
  }
  __device__ __forceinline__ float get(int j) const {
    const uint32_t w = j < 2 ? r.x : j < 4 ? r.y : j < 6 ? r.z : r.w;
    return (j & 1) ? bf16_hi(w) : bf16_lo(w);
  }
};

template <>
struct GradVec<true> {  // 8 fp32 = two 16-byte vectors
  float4 a, b;
  __device__ __forceinline__ void load(const void* p, int64_t e0) {
    const float4* q = reinterpret_cast<const float4*>(static_cast<const float*>(p) + e0);
    a = ld_grad(q);
    b = ld_grad(q + 1);
  }
  __device__ __forceinline__ float get(int j) const {
    const float4& h = j < 4 ? a : b;
    const int i = j & 3;
    return i == 0 ? h.x : i == 1 ? h.y : i == 2 ? h.z : h.w;
  }
};

template <bool GF32>
__device__ __forceinline__ float grad_scalar(const void* p, int64_t e) {
  if (GF32) return ld_grad(static_cast<const float*>(p) + e);
  return bf16_to_f32(ld_grad(static_cast<const uint16_t*>(p) + e));
}

// Sum over ranks of 8 consecutive elements.  The accumulator starts at -0.0,
// the exact identity of IEEE addition (-0 + x == x for every x, +0 included),
// so the result equals g_0 + g_1 + ... + g_{N-1} evaluated from g_0.
template <int NT, int CAP, bool GF32, bool ABF16>
__device__ __forceinline__ void sum_grads8(const StepArgs<CAP>& a, int world, int64_t e0,
                                           float acc[8]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = -0.0f;
  if (a.gvec) {
    // Ranks in groups: all of a group's 16-byte loads are issued before any
    // of them is consumed.  The any-N instance (NT = 0) takes groups of 4
    // (2 for fp32 gradients), so that it fits two blocks per SM without
    // spilling (see zero_adam_step_any_kernel).
    constexpr int GMAX = GF32 ? 8 : 16;
    constexpr int G = (NT > 0 && NT <= GMAX) ? NT : NT > 0 ? 8 : GF32 ? 2 : 4;
#pragma unroll 1
    for (int k0 = 0; k0 < world; k0 += G) {
      GradVec<GF32> r[G];
#pragma unroll
      for (int j = 0; j < G; ++j)
        if (NT > 0 || k0 + j < world) r[j].load(a.g[k0 + j], e0);
#pragma unroll
      for (int j = 0; j < G; ++j)
        if (NT > 0 || k0 + j < world) {
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = acc_add<ABF16>(acc[i], r[j].get(i));
        }
    }
  } else {
#pragma unroll 1
    for (int k = 0; k < world; ++k) {
      float x[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = grad_scalar<GF32>(a.g[k], e0 + j);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = acc_add<ABF16>(acc[j], x[j]);
    }
  }
}

__device__ __forceinline__ void load_f32x8(const float* p, bool vec, float x[8]) {
  if (vec) {
    const float4 a = ld_state(reinterpret_cast<const float4*>(p));
    const float4 b = ld_state(reinterpret_cast<const float4*>(p) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = ld_state(p + j);
  }
}

__device__ __forceinline__ void store_f32x8(float* p, bool vec, const float x[8]) {
  if (vec) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(x[0], x[1], x[2], x[3]));
    __stcs(reinterpret_cast<float4*>(p) + 1, make_float4(x[4], x[5], x[6], x[7]));
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) __stcs(p + j, x[j]);
  }
}

__device__ __forceinline__ void store_bf16x8_rn(uint16_t* p, bool vec, const float x[8]) {
  if (vec) {
    const uint4 r = make_uint4(pack_bf16x2_rn(x[0], x[1]), pack_bf16x2_rn(x[2], x[3]),
                               pack_bf16x2_rn(x[4], x[5]), pack_bf16x2_rn(x[6], x[7]));
    __stcs(reinterpret_cast<uint4*>(p), r);
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) __stcs(reinterpret_cast<unsigned short*>(p) + j, f32_to_bf16_rn(x[j]));
  }
}

// One element, no vector access (range head and tail).
template <int NT, int CAP, bool GF32, bool ABF16>
__device__ __forceinline__ void step_element(const StepArgs<CAP>& a, int world, int64_t e) {
  float acc = -0.0f;
#pragma unroll 1
  for (int k = 0; k < world; ++k) acc = acc_add<ABF16>(acc, grad_scalar<GF32>(a.g[k], e));
  float w = ld_state(a.master + e), mm = ld_state(a.m + e), vv = ld_state(a.v + e);
  adam_element<kPow2<NT>>(acc, a.s, w, mm, vv);
  a.master[e] = w;
  a.m[e] = mm;
  a.v[e] = vv;
  a.param[e] = f32_to_bf16_rn(w);
}

// The step over the range: 8 consecutive elements per thread and iteration
// (grid-stride), the unaligned head and the tail one element per thread.
template <int NT, int CAP, bool GF32, bool ABF16>
__device__ __forceinline__ void step_range(const StepArgs<CAP>& a) {
  const int world = NT > 0 ? NT : a.world;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;

  for (int64_t q = tid; q < a.nvec; q += nthreads) {
    const int64_t e0 = a.head + 8 * q;
    float acc[8], w[8], mm[8], vv[8];
    sum_grads8<NT, CAP, GF32, ABF16>(a, world, e0, acc);
    load_f32x8(a.master + e0, a.svec, w);
    load_f32x8(a.m + e0, a.svec, mm);
    load_f32x8(a.v + e0, a.svec, vv);
#pragma unroll
    for (int j = 0; j < 8; ++j) adam_element<kPow2<NT>>(acc[j], a.s, w[j], mm[j], vv[j]);
    store_f32x8(a.master + e0, a.svec, w);
    store_f32x8(a.m + e0, a.svec, mm);
    store_f32x8(a.v + e0, a.svec, vv);
    store_bf16x8_rn(a.param + e0, a.pvec, w);
  }
  for (int64_t e = tid; e < a.head; e += nthreads) step_element<NT, CAP, GF32, ABF16>(a, world, e);
  for (int64_t e = a.head + 8 * a.nvec + tid; e < a.n; e += nthreads)
    step_element<NT, CAP, GF32, ABF16>(a, world, e);
}

// The fixed-N instances (N = 1, 2, 4, ..., 64): the compiler's own register
// choice, 56-61 registers, fits two blocks of 512 threads per SM.  (A bound
// of one block per SM let it take 76-94 registers in several of them, which
// then fit one block per SM and ran up to 3 % slower.)
template <int NT, int CAP, bool GF32, bool ABF16>
__global__ void __launch_bounds__(kThreads)
    zero_adam_step_kernel(const __grid_constant__ StepArgs<CAP> a) {
  step_range<NT, CAP, GF32, ABF16>(a);
}

// The any-N instance (N read at run time, the rank loop not unrolled), held
// to two blocks per SM (at most 64 registers): with rank groups of 8 it used
// 86 registers, fit one block per SM and streamed 0.64-0.87 of the copy peak
// at N = 3, 5, 6, 7, 12, 48 on GB300, against 0.94-1.00 with groups of 4 at
// two blocks per SM.
template <int CAP, bool GF32, bool ABF16>
__global__ void __launch_bounds__(kThreads, 2)
    zero_adam_step_any_kernel(const __grid_constant__ StepArgs<CAP> a) {
  step_range<0, CAP, GF32, ABF16>(a);
}

// Status word of the staged kernels' bounded waits (read and cleared by
// zero_device_status): nonzero once a wait has given up.
__device__ int g_step_status;

// ---------------------------------------------------------------------------
// TMA-staged gradients, register-staged state: the variant for N >= 5 (bf16
// gradients, fp32 sum, buffers 16-byte aligned).  One CTA per SM.  A tile of
// TILE = CW*32*EPT elements is reduced over the ranks in groups of G: ring
// stage k holds G ranks' gradient tiles (G bulk copies of TILE*2 bytes,
// cp.async.bulk on the TMA engine), so a tile passes through ceil(N/G) stages
// and the ring depth in bytes does not grow with N.  Warp 0 is the producer:
// lane 0 arms the stage's mbarrier with its byte count, then lane r issues
// rank r's copy, so N copies per tile go out in parallel instead of from one
// thread.  The CW consumer warps' threads each own EPT consecutive elements of
// the tile: they load their master, m and v into registers (16- or 8-byte
// loads) before they wait for the first group, so those loads overlap the
// gradient copies; they add the groups in rank order from shared memory, hand
// each stage back, and after the last group run adam_element_uniform and
// store.  Every wait is bounded by about one second of the GPU's global timer;
// a wait that gives up records a nonzero status in g_step_status (read by
// zero_device_status), the producer waits (bounded) for the copies it issued,
// and every thread returns.
//
// Two shapes, chosen by N (measured on GB300 against the register-staged
// kernel, bit-exact in every case): G = 8, EPT = 4, 22 consumer warps, 3
// stages of 44 KB for 5 <= N < 40 (against the register-staged kernel's
// any-N instance, 2e8 elements: N = 5 0.958 vs 0.956 of the copy peak, with a
// tenth of the gradients exactly zero 0.906 vs 0.878; N = 12 1.065 vs 1.023;
// N = 32: 0.93 -> 1.03 on a 16.8M-element shard; at N = 8
// 1.03-1.05 with and without exact-zero gradients; at N = 16 1.058 on the 1.3B
// workload, level with an earlier kernel that also staged master/m/v through
// the ring behind 8 consumer warps, which fell to 0.86 when 10 % of the
// gradients were exact zeros while this one held 1.06); G = 32, EPT = 2, 16
// consumer warps, 3 stages of 64 KB for N >= 40 (N = 48: 1.022 vs 0.943 for the
// any-N instance; N = 64: 0.92 -> 0.975 on a 3.16M-element shard, 0.99 -> 1.00
// on 8.4M).

template <int CAP>
struct GradStagedArgs {
  const uint16_t* g[CAP];  // rank k's gradient, at the range's first element
  float* master;
  float* m;
  float* v;
  uint16_t* param;
  int64_t n;      // elements in the range
  int64_t nbody;  // multiple of 8: [0, nbody) through the ring, [nbody, n) scalar
  int32_t world;
  int32_t withhold;  // test hook: the producer issues no copies, so every wait runs out
  AdamScalars s;
};

// EPT consecutive bf16 gradients of one rank from shared memory, added to acc.
template <int EPT>
__device__ __forceinline__ void add_smem_bf16(float* acc, const uint8_t* p) {
  if constexpr (EPT == 2) {
    const uint32_t q = *reinterpret_cast<const uint32_t*>(p);
    acc[0] = __fadd_rn(acc[0], bf16_lo(q));
    acc[1] = __fadd_rn(acc[1], bf16_hi(q));
  } else if constexpr (EPT == 4) {
    const uint2 q = *reinterpret_cast<const uint2*>(p);
    acc[0] = __fadd_rn(acc[0], bf16_lo(q.x));
    acc[1] = __fadd_rn(acc[1], bf16_hi(q.x));
    acc[2] = __fadd_rn(acc[2], bf16_lo(q.y));
    acc[3] = __fadd_rn(acc[3], bf16_hi(q.y));
  } else {
    accumulate_bf16x8(acc, *reinterpret_cast<const uint4*>(p));
  }
}

// EPT (2, 4 or 8) fp32 state values: one or two vector loads / stores.
template <int EPT>
__device__ __forceinline__ void load_state_vec(const float* p, float* x) {
  if constexpr (EPT == 2) {
    const float2 q = ld_state(reinterpret_cast<const float2*>(p));
    x[0] = q.x;
    x[1] = q.y;
  } else {
#pragma unroll
    for (int j = 0; j < EPT; j += 4) {
      const float4 q = ld_state(reinterpret_cast<const float4*>(p + j));
      x[j] = q.x;
      x[j + 1] = q.y;
      x[j + 2] = q.z;
      x[j + 3] = q.w;
    }
  }
}
template <int EPT>
__device__ __forceinline__ void store_state_vec(float* p, const float* x) {
  if constexpr (EPT == 2) {
    __stcs(reinterpret_cast<float2*>(p), make_float2(x[0], x[1]));
  } else {
#pragma unroll
    for (int j = 0; j < EPT; j += 4)
      __stcs(reinterpret_cast<float4*>(p + j), make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]));
  }
}
template <int EPT>
__device__ __forceinline__ void store_param_vec(uint16_t* p, const float* x) {
  if constexpr (EPT == 2) {
    __stcs(reinterpret_cast<unsigned int*>(p), pack_bf16x2_rn(x[0], x[1]));
  } else if constexpr (EPT == 4) {
    __stcs(reinterpret_cast<uint2*>(p),
           make_uint2(pack_bf16x2_rn(x[0], x[1]), pack_bf16x2_rn(x[2], x[3])));
  } else {
    store_bf16x8_rn(p, true, x);
  }
}

template <int G, int EPT, int CW, int STAGES>
struct GradStagedShape {
  static constexpr int kTile = CW * 32 * EPT;            // elements per tile
  static constexpr int64_t kGradBytes = int64_t{kTile} * 2;  // one rank's tile
  static constexpr int64_t kStage = G * kGradBytes;      // one stage: G ranks
  static constexpr size_t kSmem = static_cast<size_t>(STAGES) * kStage;
  static_assert(G >= 1 && G <= 32, "one producer lane per rank of a group");
  static_assert(EPT == 2 || EPT == 4 || EPT == 8, "2, 4 or 8 elements per thread");
  static_assert(kTile % 8 == 0, "tiles start on 16-byte boundaries");
  static_assert(kSmem <= 227 * 1024, "ring exceeds one CTA's shared memory");
};

// The producer warp of the gradient-staged step (all 32 lanes).
template <int G, int EPT, int CW, int STAGES, int CAP>
__device__ void grad_stage_producer(const GradStagedArgs<CAP>& a, uint8_t* ring, uint64_t* full,
                                    uint64_t* empty, int lane) {
  using Shape = GradStagedShape<G, EPT, CW, STAGES>;
  constexpr int kTile = Shape::kTile;
  const int world = a.world;
  const int ngroups = (world + G - 1) / G;
  const int64_t ntiles = (a.nbody + kTile - 1) / kTile;
  int64_t k = 0;  // stages issued
  bool ok = true;
  for (int64_t tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
    const int64_t e0 = tile * kTile;
    int64_t cnt = a.nbody - e0;
    if (cnt > kTile) cnt = kTile;
    const uint32_t gbytes = static_cast<uint32_t>(cnt * 2);  // a multiple of 16
    for (int grp = 0; grp < ngroups; ++grp) {
      const int s = static_cast<int>(k % STAGES);
      if (k >= STAGES) {
        int got = 1;
        if (lane == 0)
          got = mbar_wait(&empty[s], static_cast<uint32_t>((k / STAGES - 1) & 1)) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, got, 0)) {
          ok = false;
          break;
        }
      }
      if (!a.withhold) {
        const int r0 = grp * G;
        const int nr = world - r0 < G ? world - r0 : G;
        uint8_t* st = ring + s * Shape::kStage;
        if (lane == 0) mbar_expect_tx(&full[s], gbytes * nr);
        __syncwarp();
        if (lane < nr)
          bulk_load(st + lane * Shape::kGradBytes, a.g[r0 + lane] + e0, gbytes, &full[s]);
      }
      ++k;
    }
  }
  if (!ok && lane == 0) {
    atomicExch(&g_step_status, 1);
    const int64_t first = k > STAGES ? k - STAGES : 0;
    for (int64_t j = first; j < k && !a.withhold; ++j)
      mbar_wait(&full[j % STAGES], static_cast<uint32_t>((j / STAGES) & 1));
  }
}

// The consumer warps of the gradient-staged step; t = thread index among them.
// False if a wait gave up (the step is incomplete; nothing more is written).
template <int G, int EPT, int CW, int STAGES, int CAP>
__device__ bool grad_stage_consumer(const GradStagedArgs<CAP>& a, const uint8_t* ring,
                                    uint64_t* full, uint64_t* empty, int t, int lane) {
  using Shape = GradStagedShape<G, EPT, CW, STAGES>;
  constexpr int kTile = Shape::kTile;
  const int world = a.world;
  const int ngroups = (world + G - 1) / G;
  const int64_t ntiles = (a.nbody + kTile - 1) / kTile;
  int64_t k = 0;  // stages consumed
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t e0 = tile * kTile + static_cast<int64_t>(EPT) * t;
    const bool in = e0 < a.nbody;  // e0 a multiple of EPT, nbody of 8: all EPT are in
    float acc[EPT], w[EPT], mm[EPT], vv[EPT];
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      acc[j] = -0.0f;
      w[j] = mm[j] = vv[j] = 0.0f;
    }
    if (in) {
      load_state_vec<EPT>(a.master + e0, w);
      load_state_vec<EPT>(a.m + e0, mm);
      load_state_vec<EPT>(a.v + e0, vv);
    }
    for (int grp = 0; grp < ngroups; ++grp, ++k) {
      const int s = static_cast<int>(k % STAGES);
      if (!mbar_wait(&full[s], static_cast<uint32_t>((k / STAGES) & 1))) {
        atomicExch(&g_step_status, 2);
        return false;
      }
      const int nr = world - grp * G < G ? world - grp * G : G;
      const uint8_t* st = ring + s * Shape::kStage + 2 * EPT * t;
      if (in) {
#pragma unroll
        for (int r = 0; r < G; ++r)
          if (r < nr) add_smem_bf16<EPT>(acc, st + r * Shape::kGradBytes);
      }
      // every lane has read its slice of stage s: the warp hands the stage back
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (in) {
#pragma unroll
      for (int j = 0; j < EPT; ++j) adam_element_uniform(acc[j], a.s, w[j], mm[j], vv[j]);
      store_state_vec<EPT>(a.master + e0, w);
      store_state_vec<EPT>(a.m + e0, mm);
      store_state_vec<EPT>(a.v + e0, vv);
      store_param_vec<EPT>(a.param + e0, w);
    }
  }
  return true;
}

// The last few (< 8) elements of a staged range, one per thread t of block 0.
template <int CAP>
__device__ void staged_tail(const GradStagedArgs<CAP>& a, int t) {
  if (blockIdx.x != 0 || a.nbody + t >= a.n) return;
  const int64_t e = a.nbody + t;
  float acc = -0.0f;
  for (int r = 0; r < a.world; ++r) acc = __fadd_rn(acc, bf16_to_f32(ld_grad(a.g[r] + e)));
  float w = ld_state(a.master + e), mm = ld_state(a.m + e), vv = ld_state(a.v + e);
  adam_element<0>(acc, a.s, w, mm, vv);
  a.master[e] = w;
  a.m[e] = mm;
  a.v[e] = vv;
  a.param[e] = f32_to_bf16_rn(w);
}

template <int G, int EPT, int CW, int STAGES, int CAP>
__global__ void __launch_bounds__(CW * 32 + 32, 1)
    zero_adam_step_tma_grad_kernel(const __grid_constant__ GradStagedArgs<CAP> a) {
  extern __shared__ __align__(1024) uint8_t ring[];
  __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES];
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], CW);
    }
    mbar_init_fence();
  }
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (warp == 0) {
    grad_stage_producer<G, EPT, CW, STAGES, CAP>(a, ring, full, empty, lane);
    return;
  }
  const int t = threadIdx.x - 32;
  if (grad_stage_consumer<G, EPT, CW, STAGES, CAP>(a, ring, full, empty, t, lane))
    staged_tail(a, t);
}

template <int G, int EPT, int CW, int STAGES, int CAP>
bool launch_tma_grad_shape(const StepLaunch& L, int64_t nbody, cudaError_t* err) {
  using Shape = GradStagedShape<G, EPT, CW, STAGES>;
  static std::mutex mu;
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!configured[dev]) {
      if (cudaFuncSetAttribute(zero_adam_step_tma_grad_kernel<G, EPT, CW, STAGES, CAP>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(Shape::kSmem)) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
      }
      configured[dev] = true;
    }
  }
  int sms = 0;
  if (device_sm_count(&sms) != 0) return false;
  GradStagedArgs<CAP> t;
  for (int k = 0; k < L.world; ++k) t.g[k] = static_cast<const uint16_t*>(L.grads[k]);
  for (int k = L.world; k < CAP; ++k) t.g[k] = nullptr;
  t.master = L.master;
  t.m = L.m;
  t.v = L.v;
  t.param = L.param;
  t.n = L.n;
  t.nbody = nbody;
  t.world = L.world;
  t.withhold = L.withhold;
  t.s = L.s;
  const int64_t ntiles = (nbody + Shape::kTile - 1) / Shape::kTile;
  const int grid = static_cast<int>(ntiles < sms ? ntiles : sms);
  zero_adam_step_tma_grad_kernel<G, EPT, CW, STAGES, CAP>
      <<<grid, CW * 32 + 32, Shape::kSmem, L.stream>>>(t);
  *err = cudaGetLastError();
  return true;
}

// The gradient-staged kernel for N >= 5 (not 16), when every buffer is
// 16-byte aligned at the range's first element.  Returns false when it does
// not apply.
bool launch_tma_grad(const StepLaunch& L, int32_t head, int64_t nvec, bool all_vec,
                     cudaError_t* err) {
  if (!(head == 0 && all_vec) || nvec < 1 || L.world < 5) return false;
  const int64_t nbody = 8 * nvec;
  if (L.world < 40) return launch_tma_grad_shape<8, 4, 22, 3, 64>(L, nbody, err);
  if (L.world <= 64) return launch_tma_grad_shape<32, 2, 16, 3, 64>(L, nbody, err);
  return launch_tma_grad_shape<32, 2, 16, 3, kTableRuntime>(L, nbody, err);
}

// ---------------------------------------------------------------------------
// ZeRO-3 unit step ("ZeRO and FSDP" -> "ZeRO-3 and FSDP"): the unit's
// all-gather of the N bf16 parameter shards and one rank's fused step on its
// shard, in one launch.  The step never reads the gathered unit and the
// gather never reads what the step writes (the host checks that the buffers
// are disjoint), so the two can run side by side: every CTA (one per SM) runs
// the gather's TMA copy ring in warp 1 (its chunks blockIdx.x + i*gridDim.x)
// beside its share of the step's tiles (warp 0 the gradient producer, the CW
// warps from 2 on the consumers).  Each part pays no launch of its own, and a
// small unit's gather and step overlap their ramps and DRAM round trips
// instead of running one after the other.  For N <= 4 the consumers read the
// gradients straight from global memory (GREG: no gradient ring; at small N
// the register-staged form measured faster).  Results are bit for bit those
// of zero3_unit_gather followed by zero_adam_step.

template <int CAP>
struct FlatGatherPart {
  const uint16_t* src[CAP];  // the N parameter shards
  uint16_t* full;
  int64_t numel;
  int64_t u8;     // numel rounded down to a multiple of 8: [0, u8) moves by TMA
  int64_t shard;  // a multiple of 8
};

template <int CAP>
struct UnitStepArgs {
  GradStagedArgs<CAP> step;
  FlatGatherPart<CAP> gather;
};

// Register-staged consumers for the fused kernel at N <= 4: tiles of
// CW*32*EPT elements, each thread loads its EPT gradients of every rank and
// its state, sums in rank order, updates and stores.
template <int EPT, int CW, int CAP>
__device__ void grad_reg_consumer(const GradStagedArgs<CAP>& a, int t) {
  constexpr int kTile = CW * 32 * EPT;
  static_assert(EPT == 8, "one 16-byte gradient load per rank");
  const int64_t ntiles = (a.nbody + kTile - 1) / kTile;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t e0 = tile * kTile + static_cast<int64_t>(EPT) * t;
    if (e0 >= a.nbody) continue;
    uint4 r[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (k < a.world) r[k] = ld_grad(reinterpret_cast<const uint4*>(a.g[k] + e0));
    float w[8], mm[8], vv[8], acc[8];
    load_state_vec<8>(a.master + e0, w);
    load_state_vec<8>(a.m + e0, mm);
    load_state_vec<8>(a.v + e0, vv);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = -0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (k < a.world) accumulate_bf16x8(acc, r[k]);
#pragma unroll
    for (int j = 0; j < 8; ++j) adam_element<0>(acc[j], a.s, w[j], mm[j], vv[j]);
    store_state_vec<8>(a.master + e0, w);
    store_state_vec<8>(a.m + e0, mm);
    store_state_vec<8>(a.v + e0, vv);
    store_param_vec<8>(a.param + e0, w);
  }
}

template <int G, int EPT, int CW, int STAGES, int SLOTS, int CAP, bool GREG>
struct UnitStepShape {
  using Step = GradStagedShape<G, EPT, CW, STAGES>;
  static constexpr size_t kStepRing = GREG ? 0 : Step::kSmem;
  static constexpr size_t kSmem = kStepRing + static_cast<size_t>(SLOTS) * kSlotBytes;
  static_assert(kSmem + 1024 <= 227 * 1024, "rings exceed one CTA's shared memory");
};

template <int G, int EPT, int CW, int STAGES, int SLOTS, int CAP, bool GREG>
__global__ void __launch_bounds__(CW * 32 + 64, 1)
    zero3_unit_step_kernel(const __grid_constant__ UnitStepArgs<CAP> a) {
  using Shape = UnitStepShape<G, EPT, CW, STAGES, SLOTS, CAP, GREG>;
  extern __shared__ __align__(1024) uint8_t ring[];  // [step ring][gather ring]
  __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], gbar[SLOTS];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], CW);
    }
    for (int s = 0; s < SLOTS; ++s) mbar_init(&gbar[s], 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (warp == 0) {
    if (!GREG) grad_stage_producer<G, EPT, CW, STAGES, CAP>(a.step, ring, full, empty, lane);
    return;
  }
  if (warp == 1) {
    const FlatGatherPart<CAP>& g = a.gather;
    // the unit's last (< 8) elements, lanes of block 0
    if (blockIdx.x == 0 && g.u8 + lane < g.numel && !a.step.withhold) {
      const int64_t e = g.u8 + lane;
      const int64_t r = e / g.shard;
      g.full[e] = g.src[r][e - r * g.shard];
    }
    const int64_t nchunks = flat_chunks(g.u8);
    if (lane != 0 || blockIdx.x >= nchunks) return;
    const int64_t mine = (nchunks - blockIdx.x + gridDim.x - 1) / gridDim.x;
    FlatLayout<FlatGatherPart<CAP>> layout{g};
    ring_copy<SLOTS>(layout, mine, ring + Shape::kStepRing, gbar, a.step.withhold != 0,
                     &g_step_status);
    return;
  }
  const int t = threadIdx.x - 64;
  if constexpr (GREG) {
    grad_reg_consumer<EPT, CW, CAP>(a.step, t);
    staged_tail(a.step, t);
  } else {
    if (grad_stage_consumer<G, EPT, CW, STAGES, CAP>(a.step, ring, full, empty, t, lane))
      staged_tail(a.step, t);
  }
}

template <int G, int EPT, int CW, int STAGES, int SLOTS, int CAP, bool GREG>
bool launch_unit_step_shape(const GatherLaunch& GL, const StepLaunch& L, int64_t nbody,
                            cudaError_t* err) {
  using Shape = UnitStepShape<G, EPT, CW, STAGES, SLOTS, CAP, GREG>;
  auto kernel = zero3_unit_step_kernel<G, EPT, CW, STAGES, SLOTS, CAP, GREG>;
  static std::mutex mu;
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!configured[dev]) {
      if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(Shape::kSmem)) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
      }
      configured[dev] = true;
    }
  }
  int sms = 0;
  if (device_sm_count(&sms) != 0) return false;
  UnitStepArgs<CAP> u;
  GradStagedArgs<CAP>& t = u.step;
  for (int k = 0; k < L.world; ++k) t.g[k] = static_cast<const uint16_t*>(L.grads[k]);
  for (int k = L.world; k < CAP; ++k) t.g[k] = nullptr;
  t.master = L.master;
  t.m = L.m;
  t.v = L.v;
  t.param = L.param;
  t.n = L.n;
  t.nbody = nbody;
  t.world = L.world;
  t.withhold = L.withhold;
  t.s = L.s;
  FlatGatherPart<CAP>& g = u.gather;
  for (int k = 0; k < GL.world; ++k) g.src[k] = GL.shards[k];
  for (int k = GL.world; k < CAP; ++k) g.src[k] = nullptr;
  g.full = GL.full;
  g.numel = GL.numel;
  g.u8 = GL.numel & ~static_cast<int64_t>(7);
  g.shard = GL.shard;
  constexpr int64_t kTile = GREG ? int64_t{CW} * 32 * EPT : Shape::Step::kTile;
  int64_t work = (nbody + kTile - 1) / kTile;
  const int64_t nchunks = flat_chunks(g.u8);
  if (nchunks > work) work = nchunks;
  const int grid = static_cast<int>(work < sms ? (work < 1 ? 1 : work) : sms);
  kernel<<<grid, CW * 32 + 64, Shape::kSmem, L.stream>>>(u);
  *err = cudaGetLastError();
  return true;
}

// Resident blocks per SM of a kernel on the current device (cached).
int blocks_per_sm(const void* kernel) {
  static std::mutex mu;
  static std::unordered_map<const void*, int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache[dev].find(kernel);
  if (it != cache[dev].end()) return it->second;
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, kThreads, 0) != cudaSuccess ||
      nb < 1)
    nb = 1;
  cache[dev][kernel] = nb;
  return nb;
}

// Element residue of an address within its 16-byte line.
inline int residue(const void* p, int esize) {
  return static_cast<int>((reinterpret_cast<uintptr_t>(p) / esize) % (16 / esize));
}

template <int NT, int CAP, bool GF32, bool ABF16>
cudaError_t launch_world(const StepLaunch& L) {
  StepArgs<CAP> a;
  for (int k = 0; k < L.world; ++k) a.g[k] = L.grads[k];
  for (int k = L.world; k < CAP; ++k) a.g[k] = nullptr;
  a.master = L.master;
  a.m = L.m;
  a.v = L.v;
  a.param = L.param;
  a.n = L.n;
  a.world = L.world;
  a.s = L.s;

  // Pick the body's start (head in 0..7) that lets the most bytes per element
  // move as 16-byte vectors: all gradients together (N * 2 or 4 B), the fp32
  // state (24 B), the bf16 parameters (2 B).  Buffers from cudaMalloc used
  // whole are all aligned at head = 0.
  const int gsize = GF32 ? 4 : 2;
  const int gmod = 16 / gsize;
  int rg = residue(L.grads[0], gsize);
  for (int k = 1; k < L.world; ++k)
    if (residue(L.grads[k], gsize) != rg) rg = -1;
  int rs = residue(L.master, 4);
  if (residue(L.m, 4) != rs || residue(L.v, 4) != rs) rs = -1;
  const int rp = residue(L.param, 2);
  int best_h = 0, best_score = -1;
  for (int h = 0; h < 8; ++h) {
    const int score = ((rg >= 0 && (rg + h) % gmod == 0) ? gsize * L.world : 0) +
                      ((rs >= 0 && (rs + h) % 4 == 0) ? 24 : 0) + (((rp + h) % 8 == 0) ? 2 : 0);
    if (score > best_score) {
      best_score = score;
      best_h = h;
    }
  }
  int64_t head = best_h;
  if (head > L.n) head = L.n;
  a.head = static_cast<int32_t>(head);
  a.nvec = (L.n - head) / 8;
  a.gvec = (rg >= 0 && (rg + best_h) % gmod == 0);
  a.svec = (rs >= 0 && (rs + best_h) % 4 == 0);
  a.pvec = ((rp + best_h) % 8 == 0);

  if constexpr (!GF32 && !ABF16) {
    cudaError_t err = cudaSuccess;
    if (launch_tma_grad(L, a.head, a.nvec, a.gvec && a.svec && a.pvec, &err)) return err;
  }

  const void* kern;
  if constexpr (NT == 0)
    kern = reinterpret_cast<const void*>(&zero_adam_step_any_kernel<CAP, GF32, ABF16>);
  else
    kern = reinterpret_cast<const void*>(&zero_adam_step_kernel<NT, CAP, GF32, ABF16>);
  int sms = 0;
  if (device_sm_count(&sms) != 0) return cudaErrorNoDevice;
  const int64_t cap = static_cast<int64_t>(sms) * blocks_per_sm(kern);
  int64_t blocks = (a.nvec + kThreads - 1) / kThreads;
  if (blocks < 1) blocks = 1;
  if (blocks > cap) blocks = cap;
  if constexpr (NT == 0)
    zero_adam_step_any_kernel<CAP, GF32, ABF16>
        <<<static_cast<unsigned>(blocks), kThreads, 0, L.stream>>>(a);
  else
    zero_adam_step_kernel<NT, CAP, GF32, ABF16>
        <<<static_cast<unsigned>(blocks), kThreads, 0, L.stream>>>(a);
  return cudaGetLastError();
}

template <bool GF32, bool ABF16>
cudaError_t launch_variant(const StepLaunch& L) {
  switch (L.world) {
    case 1: return launch_world<1, 1, GF32, ABF16>(L);
    case 2: return launch_world<2, 2, GF32, ABF16>(L);
    case 4: return launch_world<4, 4, GF32, ABF16>(L);
    case 8: return launch_world<8, 8, GF32, ABF16>(L);
    case 16: return launch_world<16, 16, GF32, ABF16>(L);
    case 32: return launch_world<32, 32, GF32, ABF16>(L);
    case 64: return launch_world<64, 64, GF32, ABF16>(L);
    default: return launch_world<0, kTableRuntime, GF32, ABF16>(L);
  }
}

// Largest unit (gather bytes + step bytes) that takes the single launch.
// Measured on GB300 against the gather and the step as two launches, units
// of 2^22..2^27 elements with the L2 flushed: at N = 2 and 8 the single launch
// takes 0.71-0.87 of the time up to 320 MB and 0.95-0.98 at 620 MB, and
// 1.01-1.03 at 1.2 GB; at N = 32 and 64 0.65-0.81 up to 460 MB.  Past these
// sizes each kernel alone streams at its own best and the launch cost is
// amortised, while inside the single launch the gather's ring falls behind
// the step's consumers and finishes alone.
constexpr int64_t kFusedMaxBytes = int64_t{512} << 20;

// The fused unit step when both parts can run on the TMA engine: the gather's
// shard a multiple of 8 elements, and every buffer of both parts 16-byte
// aligned at its first element; bf16 gradients, fp32 sum; a unit below the
// size limit above.
bool launch_unit_step_fused(const GatherLaunch& GL, const StepLaunch& L, cudaError_t* err) {
  if (L.grad_f32 || L.acc_bf16 || L.n < 8 || GL.numel < 8 || GL.shard % 8 != 0) return false;
  const int64_t bytes = 4 * GL.numel + (2 * static_cast<int64_t>(L.world) + 26) * L.n;
  if (bytes > kFusedMaxBytes) return false;
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  bool ok = a16(GL.full) && a16(L.master) && a16(L.m) && a16(L.v) && a16(L.param);
  for (int k = 0; k < GL.world && ok; ++k) ok = a16(GL.shards[k]);
  for (int k = 0; k < L.world && ok; ++k) ok = a16(L.grads[k]);
  if (!ok) return false;
  const int64_t nbody = L.n & ~static_cast<int64_t>(7);
  // N >= 24: a two-stage step ring leaves room for four gather slots (measured
  // against three stages and two slots: 2^24-element units at N = 64 0.0146 vs
  // 0.0209 ms, at N = 32 0.0154 vs 0.0168 with the N < 24 shape).
  if (L.world <= 4) return launch_unit_step_shape<1, 8, 24, 1, 4, 64, true>(GL, L, nbody, err);
  if (L.world < 24) return launch_unit_step_shape<8, 4, 22, 3, 4, 64, false>(GL, L, nbody, err);
  if (L.world <= 64) return launch_unit_step_shape<32, 2, 16, 2, 4, 64, false>(GL, L, nbody, err);
  return launch_unit_step_shape<32, 2, 16, 2, 4, kTableRuntime, false>(GL, L, nbody, err);
}

}  // namespace

cudaError_t launch_unit_step(const GatherLaunch& GL, const StepLaunch& L) {
  (void)cudaGetLastError();  // launch errors below are this call's own
  if (L.n <= 0) return launch_unit_gather(GL);
  cudaError_t err = cudaSuccess;
  if (launch_unit_step_fused(GL, L, &err)) return err;
  err = launch_unit_gather(GL);
  if (err != cudaSuccess) return err;
  return launch_adam_step(L);
}

namespace {
__device__ int g_step_status_taken;

// Reads and clears the status word in one atomic exchange, so that a flag a
// kernel still running on another stream sets is either taken now or kept
// for the next read, never lost between a read and a separate clear.
__global__ void take_step_status_kernel() {
  g_step_status_taken = atomicExch(&g_step_status, 0);
}
}  // namespace

int read_and_clear_step_status(int* status) {
  take_step_status_kernel<<<1, 1, 0, 0>>>();
  if (cudaGetLastError() != cudaSuccess) return -1;
  int v = 0;  // the copy is ordered after the kernel on the legacy default stream
  if (cudaMemcpyFromSymbol(&v, g_step_status_taken, sizeof(int)) != cudaSuccess) return -1;
  *status = v;
  return 0;
}

cudaError_t launch_adam_step(const StepLaunch& L) {
  if (L.n <= 0) return cudaSuccess;
  (void)cudaGetLastError();  // launch errors below are this call's own
  if (!L.grad_f32 && !L.acc_bf16) return launch_variant<false, false>(L);
  if (!L.grad_f32 && L.acc_bf16) return launch_variant<false, true>(L);
  if (L.grad_f32 && !L.acc_bf16) return launch_variant<true, false>(L);
  return launch_variant<true, true>(L);
}

}  // namespace zeroadam
