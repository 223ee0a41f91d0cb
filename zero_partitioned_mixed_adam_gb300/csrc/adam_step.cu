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
// the SM count) and uses no tensor cores.  For N = 16 and N = 8 with aligned
// buffers, TMA-staged variants (bulk copies into a shared-memory ring, one
// CTA per SM) replace it.
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

#include "internal.h"
#include "tma_ops.h"

namespace zeroadam {
namespace {

constexpr int kThreads = 512;
constexpr int kTableRuntime = 1024;  // gradient-pointer table of the any-N kernel

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

__device__ __forceinline__ void unpack8(const float4 a, const float4 b, float x[8]) {
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
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
// the value the IEEE division returns.  bc1 = 1 - b1^t and bc2 = 1 - b2^t are
// > 0 (beta in [0, 1), t >= 1); the last division is skipped only when its
// denominator is > 0 (0 / 0 still goes through the division and gives NaN).
// Elements whose gradient is exactly zero every step (untouched rows, dead
// units; the GPT-2 workload's 10 % mask) keep m = v = 0, and without the
// shortcut their divisions take the slow path of the IEEE division sequence.
__device__ __forceinline__ void adam_element(float gsum, const AdamScalars& s, float& w, float& m,
                                             float& v) {
  const float g = s.pow2_world ? __fmul_rn(gsum, s.inv_world) : __fdiv_rn(gsum, s.world);
  m = __fadd_rn(__fmul_rn(m, s.b1), __fmul_rn(s.omb1, g));
  v = __fadd_rn(__fmul_rn(v, s.b2), __fmul_rn(__fmul_rn(s.omb2, g), g));
  const float m_hat = (m == 0.0f) ? m : __fdiv_rn(m, s.bc1);
  const float v_hat = (v == 0.0f) ? v : __fdiv_rn(v, s.bc2);
  const float denom = __fadd_rn(__fsqrt_rn(v_hat), s.eps);
  const float num = __fmul_rn(s.lr, m_hat);
  w = __fsub_rn(w, (num == 0.0f && denom > 0.0f) ? num : __fdiv_rn(num, denom));
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
    // of them is consumed.
    constexpr int GMAX = GF32 ? 8 : 16;
    constexpr int G = (NT > 0 && NT <= GMAX) ? NT : 8;
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
  adam_element(acc, a.s, w, mm, vv);
  a.master[e] = w;
  a.m[e] = mm;
  a.v[e] = vv;
  a.param[e] = f32_to_bf16_rn(w);
}

template <int NT, int CAP, bool GF32, bool ABF16>
__global__ void __launch_bounds__(kThreads)
    zero_adam_step_kernel(const __grid_constant__ StepArgs<CAP> a) {
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
    for (int j = 0; j < 8; ++j) adam_element(acc[j], a.s, w[j], mm[j], vv[j]);
    store_f32x8(a.master + e0, a.svec, w);
    store_f32x8(a.m + e0, a.svec, mm);
    store_f32x8(a.v + e0, a.svec, vv);
    store_bf16x8_rn(a.param + e0, a.pvec, w);
  }
  for (int64_t e = tid; e < a.head; e += nthreads) step_element<NT, CAP, GF32, ABF16>(a, world, e);
  for (int64_t e = a.head + 8 * a.nvec + tid; e < a.n; e += nthreads)
    step_element<NT, CAP, GF32, ABF16>(a, world, e);
}

// ---------------------------------------------------------------------------
// TMA-staged variant for N = 16, bf16 gradients, fp32 sum (measured faster
// than the register-staged kernel there; at N = 8 the state-staged ring leaves
// room for too few consumer warps, and zero_adam_step_tma_grad_kernel below is
// used instead).
// One CTA per SM.  Warp 0 lane 0 is the producer: for each 2048-element tile
// it issues one bulk copy (cp.async.bulk, the TMA engine) per rank's gradient
// tile and per state array into a two-stage shared-memory ring, and the
// stage's mbarrier completes when all bytes have landed.  Warps 1..8 consume:
// each thread sums its 8 elements over the ranks and runs adam_element from
// shared memory, then stores to global.  Every wait is bounded by about one
// second of the GPU's global timer; a wait that gives up records a nonzero
// status in g_step_status (read by zero_device_status), the producer waits
// (bounded) for the copies it issued, and every thread returns.

constexpr int kTmaTile = 2048;       // elements per tile
constexpr int kTmaConsumers = 256;   // 8 warps, 8 elements per thread
constexpr int kTmaStages = 2;

__device__ int g_step_status;

template <int NT>
struct TmaArgs {
  const uint16_t* g[NT];
  float* master;
  float* m;
  float* v;
  uint16_t* param;
  int64_t n;      // elements in the range
  int64_t nbody;  // multiple of 8: [0, nbody) through the ring, [nbody, n) scalar
  int32_t withhold;  // test hook: the producer issues no copies, so every wait runs out
  AdamScalars s;
};

template <int NT>
__global__ void __launch_bounds__(kTmaConsumers + 32, 1)
    zero_adam_step_tma_kernel(const __grid_constant__ TmaArgs<NT> a) {
  // stage: NT bf16 gradient tiles, then the master, m and v fp32 tiles
  constexpr int64_t kGradBytes = kTmaTile * 2;
  constexpr int64_t kStage = NT * kGradBytes + 3 * kTmaTile * 4;
  extern __shared__ __align__(1024) uint8_t ring[];
  __shared__ __align__(8) uint64_t full[kTmaStages], empty[kTmaStages];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t ntiles = (a.nbody + kTmaTile - 1) / kTmaTile;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTmaStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kTmaConsumers / 32);
    }
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == 0) {
    if (lane != 0) return;
    int64_t k = 0;
    bool ok = true;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++k) {
      const int s = static_cast<int>(k % kTmaStages);
      if (k >= kTmaStages &&
          !mbar_wait(&empty[s], static_cast<uint32_t>((k / kTmaStages - 1) & 1))) {
        ok = false;
        break;
      }
      if (a.withhold) continue;
      const int64_t e0 = tile * kTmaTile;
      int64_t cnt = a.nbody - e0;
      if (cnt > kTmaTile) cnt = kTmaTile;
      const uint32_t gbytes = static_cast<uint32_t>(cnt * 2);
      uint8_t* st = ring + s * kStage;
      mbar_expect_tx(&full[s], gbytes * NT + 3 * 2 * gbytes);
      for (int r = 0; r < NT; ++r) bulk_load(st + r * kGradBytes, a.g[r] + e0, gbytes, &full[s]);
      uint8_t* sf = st + NT * kGradBytes;
      bulk_load(sf, a.master + e0, 2 * gbytes, &full[s]);
      bulk_load(sf + kTmaTile * 4, a.m + e0, 2 * gbytes, &full[s]);
      bulk_load(sf + 2 * kTmaTile * 4, a.v + e0, 2 * gbytes, &full[s]);
    }
    if (!ok) {
      atomicExch(&g_step_status, 1);
      const int64_t first = k > kTmaStages ? k - kTmaStages : 0;
      for (int64_t j = first; j < k && !a.withhold; ++j)
        mbar_wait(&full[j % kTmaStages], static_cast<uint32_t>((j / kTmaStages) & 1));
    }
    return;
  }

  const int t = threadIdx.x - 32;
  int64_t k = 0;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++k) {
    const int s = static_cast<int>(k % kTmaStages);
    if (!mbar_wait(&full[s], static_cast<uint32_t>((k / kTmaStages) & 1))) {
      atomicExch(&g_step_status, 2);
      return;
    }
    const int64_t e0 = tile * kTmaTile + 8 * t;
    const bool in = e0 < a.nbody;  // e0 and nbody are multiples of 8
    const uint8_t* st = ring + s * kStage;
    float acc[8], w[8], mm[8], vv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = -0.0f;
    if (in) {
#pragma unroll
      for (int r = 0; r < NT; ++r)
        accumulate_bf16x8(acc, *reinterpret_cast<const uint4*>(st + r * kGradBytes + 16 * t));
      const float4* sf = reinterpret_cast<const float4*>(st + NT * kGradBytes);
      unpack8(sf[2 * t], sf[2 * t + 1], w);
      unpack8(sf[kTmaTile / 4 + 2 * t], sf[kTmaTile / 4 + 2 * t + 1], mm);
      unpack8(sf[kTmaTile / 2 + 2 * t], sf[kTmaTile / 2 + 2 * t + 1], vv);
    }
    // every lane has read its slice of stage s: the warp hands the stage back
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (in) {
#pragma unroll
      for (int j = 0; j < 8; ++j) adam_element(acc[j], a.s, w[j], mm[j], vv[j]);
      store_f32x8(a.master + e0, true, w);
      store_f32x8(a.m + e0, true, mm);
      store_f32x8(a.v + e0, true, vv);
      store_bf16x8_rn(a.param + e0, true, w);
    }
  }
  // the last few (< 8) elements of the range, one per thread of block 0
  if (blockIdx.x == 0 && a.nbody + t < a.n) {
    const int64_t e = a.nbody + t;
    float acc = -0.0f;
#pragma unroll
    for (int r = 0; r < NT; ++r) acc = __fadd_rn(acc, bf16_to_f32(ld_grad(a.g[r] + e)));
    float w = ld_state(a.master + e), mm = ld_state(a.m + e), vv = ld_state(a.v + e);
    adam_element(acc, a.s, w, mm, vv);
    a.master[e] = w;
    a.m[e] = mm;
    a.v[e] = vv;
    a.param[e] = f32_to_bf16_rn(w);
  }
}

constexpr size_t tma_smem_bytes(int nt) {
  return static_cast<size_t>(kTmaStages) * (nt * kTmaTile * 2 + 3 * kTmaTile * 4);
}

// Launch the TMA kernel when every buffer is 16-byte aligned at the range's
// first element (head == 0 with all streams vectorised).  Returns false when
// the variant does not apply.
template <int NT>
bool launch_tma(const StepLaunch& L, const StepArgs<NT>& a, cudaError_t* err) {
  if (!(a.head == 0 && a.gvec && a.svec && a.pvec) || a.nvec < 1) return false;
  static std::mutex mu;
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!configured[dev]) {
      if (cudaFuncSetAttribute(zero_adam_step_tma_kernel<NT>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(tma_smem_bytes(NT))) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
      }
      configured[dev] = true;
    }
  }
  int sms = 0;
  if (device_sm_count(&sms) != 0) return false;
  TmaArgs<NT> t;
  for (int k = 0; k < NT; ++k) t.g[k] = static_cast<const uint16_t*>(L.grads[k]);
  t.master = L.master;
  t.m = L.m;
  t.v = L.v;
  t.param = L.param;
  t.n = L.n;
  t.nbody = 8 * a.nvec;
  t.withhold = L.withhold;
  t.s = L.s;
  const int64_t ntiles = (t.nbody + kTmaTile - 1) / kTmaTile;
  const int grid = static_cast<int>(ntiles < sms ? ntiles : sms);
  zero_adam_step_tma_kernel<NT>
      <<<grid, kTmaConsumers + 32, tma_smem_bytes(NT), L.stream>>>(t);
  *err = cudaGetLastError();
  return true;
}

// ---------------------------------------------------------------------------
// TMA-staged gradients, register-staged state: the variant for N = 8, bf16
// gradients, fp32 sum.  One CTA per SM.  The producer lane bulk-copies only
// the N gradient tiles of each 3072-element tile into a three-stage ring
// (8 x 6 KB per stage).  Each of the 24 consumer warps' threads owns 4
// elements of the tile: it loads their master, m and v straight into
// registers before it waits for the stage, so those loads overlap the
// gradient copies, then sums the gradients from shared memory, runs
// adam_element and stores.  At N = 8 an element carries 42 bytes instead of
// 58, so the arithmetic per byte is higher than at N = 16: with the state
// staged too, only 8 consumer warps fit beside the ring and they fall behind
// the copies; with the gradients alone, 24 do not.  Waits are bounded as in
// the kernel above, with the same status word.

constexpr int kTgEpt = 4;                          // elements per consumer thread
constexpr int kTgConsumers = 768;                  // 24 warps
constexpr int kTgTile = kTgConsumers * kTgEpt;     // 3072 elements
constexpr int kTgStages = 3;

constexpr size_t tma_grad_smem_bytes(int nt) {
  return static_cast<size_t>(kTgStages) * nt * kTgTile * 2;
}
static_assert(tma_grad_smem_bytes(8) <= 227 * 1024, "ring exceeds one CTA's shared memory");

template <int NT>
__global__ void __launch_bounds__(kTgConsumers + 32, 1)
    zero_adam_step_tma_grad_kernel(const __grid_constant__ TmaArgs<NT> a) {
  constexpr int64_t kGradBytes = kTgTile * 2;  // one rank's gradient tile
  constexpr int64_t kStage = NT * kGradBytes;
  extern __shared__ __align__(1024) uint8_t ring[];
  __shared__ __align__(8) uint64_t full[kTgStages], empty[kTgStages];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t ntiles = (a.nbody + kTgTile - 1) / kTgTile;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTgStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kTgConsumers / 32);
    }
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == 0) {
    if (lane != 0) return;
    int64_t k = 0;
    bool ok = true;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++k) {
      const int s = static_cast<int>(k % kTgStages);
      if (k >= kTgStages &&
          !mbar_wait(&empty[s], static_cast<uint32_t>((k / kTgStages - 1) & 1))) {
        ok = false;
        break;
      }
      if (a.withhold) continue;
      const int64_t e0 = tile * kTgTile;
      int64_t cnt = a.nbody - e0;
      if (cnt > kTgTile) cnt = kTgTile;
      const uint32_t gbytes = static_cast<uint32_t>(cnt * 2);  // a multiple of 16
      uint8_t* st = ring + s * kStage;
      mbar_expect_tx(&full[s], gbytes * NT);
      for (int r = 0; r < NT; ++r) bulk_load(st + r * kGradBytes, a.g[r] + e0, gbytes, &full[s]);
    }
    if (!ok) {
      atomicExch(&g_step_status, 1);
      const int64_t first = k > kTgStages ? k - kTgStages : 0;
      for (int64_t j = first; j < k && !a.withhold; ++j)
        mbar_wait(&full[j % kTgStages], static_cast<uint32_t>((j / kTgStages) & 1));
    }
    return;
  }

  const int t = threadIdx.x - 32;
  int64_t k = 0;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++k) {
    const int s = static_cast<int>(k % kTgStages);
    const int64_t e0 = tile * kTgTile + kTgEpt * t;
    const bool in = e0 < a.nbody;  // e0 is a multiple of 4, nbody of 8: all 4 are in
    float4 w = make_float4(0.f, 0.f, 0.f, 0.f), mm = w, vv = w;
    if (in) {
      w = ld_state(reinterpret_cast<const float4*>(a.master + e0));
      mm = ld_state(reinterpret_cast<const float4*>(a.m + e0));
      vv = ld_state(reinterpret_cast<const float4*>(a.v + e0));
    }
    if (!mbar_wait(&full[s], static_cast<uint32_t>((k / kTgStages) & 1))) {
      atomicExch(&g_step_status, 2);
      return;
    }
    const uint8_t* st = ring + s * kStage;
    float acc[4] = {-0.0f, -0.0f, -0.0f, -0.0f};
    if (in) {
#pragma unroll
      for (int r = 0; r < NT; ++r) {
        const uint2 q = *reinterpret_cast<const uint2*>(st + r * kGradBytes + 2 * kTgEpt * t);
        acc[0] = __fadd_rn(acc[0], bf16_lo(q.x));
        acc[1] = __fadd_rn(acc[1], bf16_hi(q.x));
        acc[2] = __fadd_rn(acc[2], bf16_lo(q.y));
        acc[3] = __fadd_rn(acc[3], bf16_hi(q.y));
      }
    }
    // every lane has read its slice of stage s: the warp hands the stage back
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (in) {
      adam_element(acc[0], a.s, w.x, mm.x, vv.x);
      adam_element(acc[1], a.s, w.y, mm.y, vv.y);
      adam_element(acc[2], a.s, w.z, mm.z, vv.z);
      adam_element(acc[3], a.s, w.w, mm.w, vv.w);
      __stcs(reinterpret_cast<float4*>(a.master + e0), w);
      __stcs(reinterpret_cast<float4*>(a.m + e0), mm);
      __stcs(reinterpret_cast<float4*>(a.v + e0), vv);
      __stcs(reinterpret_cast<uint2*>(a.param + e0),
             make_uint2(pack_bf16x2_rn(w.x, w.y), pack_bf16x2_rn(w.z, w.w)));
    }
  }
  // the last few (< 8) elements of the range, one per thread of block 0
  if (blockIdx.x == 0 && a.nbody + t < a.n) {
    const int64_t e = a.nbody + t;
    float acc = -0.0f;
#pragma unroll
    for (int r = 0; r < NT; ++r) acc = __fadd_rn(acc, bf16_to_f32(ld_grad(a.g[r] + e)));
    float w = ld_state(a.master + e), mm = ld_state(a.m + e), vv = ld_state(a.v + e);
    adam_element(acc, a.s, w, mm, vv);
    a.master[e] = w;
    a.m[e] = mm;
    a.v[e] = vv;
    a.param[e] = f32_to_bf16_rn(w);
  }
}

// As launch_tma, for the gradient-staged kernel.
template <int NT>
bool launch_tma_grad(const StepLaunch& L, const StepArgs<NT>& a, cudaError_t* err) {
  if (!(a.head == 0 && a.gvec && a.svec && a.pvec) || a.nvec < 1) return false;
  static std::mutex mu;
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!configured[dev]) {
      if (cudaFuncSetAttribute(zero_adam_step_tma_grad_kernel<NT>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(tma_grad_smem_bytes(NT))) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
      }
      configured[dev] = true;
    }
  }
  int sms = 0;
  if (device_sm_count(&sms) != 0) return false;
  TmaArgs<NT> t;
  for (int k = 0; k < NT; ++k) t.g[k] = static_cast<const uint16_t*>(L.grads[k]);
  t.master = L.master;
  t.m = L.m;
  t.v = L.v;
  t.param = L.param;
  t.n = L.n;
  t.nbody = 8 * a.nvec;
  t.withhold = L.withhold;
  t.s = L.s;
  const int64_t ntiles = (t.nbody + kTgTile - 1) / kTgTile;
  const int grid = static_cast<int>(ntiles < sms ? ntiles : sms);
  zero_adam_step_tma_grad_kernel<NT>
      <<<grid, kTgConsumers + 32, tma_grad_smem_bytes(NT), L.stream>>>(t);
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

  if constexpr (NT == 16 && CAP == 16 && !GF32 && !ABF16) {
    cudaError_t err = cudaSuccess;
    if (launch_tma<16>(L, a, &err)) return err;
  }
  if constexpr (NT == 8 && CAP == 8 && !GF32 && !ABF16) {
    cudaError_t err = cudaSuccess;
    if (launch_tma_grad<8>(L, a, &err)) return err;
  }

  const void* kern = reinterpret_cast<const void*>(&zero_adam_step_kernel<NT, CAP, GF32, ABF16>);
  int sms = 0;
  if (device_sm_count(&sms) != 0) return cudaErrorNoDevice;
  const int64_t cap = static_cast<int64_t>(sms) * blocks_per_sm(kern);
  int64_t blocks = (a.nvec + kThreads - 1) / kThreads;
  if (blocks < 1) blocks = 1;
  if (blocks > cap) blocks = cap;
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

}  // namespace

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
