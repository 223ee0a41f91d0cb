// unit_gather.cu -- ZeRO-3 unit all-gather on sm_103a ("ZeRO and FSDP" ->
// "ZeRO-3 and FSDP": before a unit is used its complete parameters are
// all-gathered from the ranks' shards).  With the ranks emulated in one
// GPU's memory the gather is a copy of N bf16 shards into one unit buffer:
//   full[r*shard + j] = shard_r[j],  r*shard + j < numel.
// The FSDP2-style gather (row blocks of each tensor per rank) is the same copy
// in T*N runs.  Both move 4 bytes per unit element (2 read, 2 written) and are
// bound by HBM bandwidth, or for small units by launch latency.  Each has two
// kernels: a copy on the TMA engine (bulk loads into a shared-memory ring,
// bulk stores out of it) when every run starts on a 16-byte boundary, and a
// vectorised load/store copy for every other layout.
#include <mutex>
#include <unordered_map>

#include "gather_ring.h"
#include "internal.h"
#include "tma_ops.h"

namespace zeroadam {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;  // 16-byte vectors in flight per thread

template <int CAP>
struct GatherArgs {
  const uint16_t* src[CAP];
  uint16_t* full;
  int64_t numel;
  int64_t shard;
  int32_t world;
  int32_t vec;  // every shard and its destination are 16-byte aligned
};

// blockIdx.y = rank; blocks along x stride over that rank's shard.
template <int CAP>
__global__ void __launch_bounds__(kThreads)
    zero3_unit_gather_kernel(const __grid_constant__ GatherArgs<CAP> a) {
  const int r = blockIdx.y;
  const int64_t lo = static_cast<int64_t>(r) * a.shard;
  int64_t cnt = a.numel - lo;
  if (cnt > a.shard) cnt = a.shard;
  if (cnt <= 0) return;
  const uint16_t* __restrict__ src = a.src[r];
  uint16_t* __restrict__ dst = a.full + lo;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t done = 0;
  if (a.vec) {
    const int64_t nv = cnt / 8;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    int64_t q = tid;
    for (; q + (kUnroll - 1) * nthreads < nv; q += kUnroll * nthreads) {
      uint4 x[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) x[u] = __ldcs(s4 + q + u * nthreads);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) __stcs(d4 + q + u * nthreads, x[u]);
    }
    for (; q < nv; q += nthreads) __stcs(d4 + q, __ldcs(s4 + q));
    done = nv * 8;
  }
  for (int64_t j = done + tid; j < cnt; j += nthreads) dst[j] = __ldcs(src + j);
}

// ---------------------------------------------------------------------------
// The gathers on the TMA engine: one thread per CTA (one CTA per SM) moves
// its chunks through a 4-slot ring in shared memory (ring_copy, the copy
// shared with the fused unit step, gather_ring.h).  Elements that do not fill
// a 16-byte unit at the end of a run are copied with plain loads and stores.
// Measured against the load/store kernels on GB300: the same bytes and about
// the same time under ncu; back to back, the flat gather 1-3 % faster on units
// of 202M and 2^29 elements (0.93-0.98 of the copy peak) and 1.5x on 2^24,
// 2.4x on 2^20 units with the L2 warm, the row gather 3.5 % faster on a
// Llama-7B layer (0.94).  A wait that gives up records a nonzero status in
// g_gather_status (read with the step kernels' word by zero_device_status).

__device__ int g_gather_status;

// Flat gather: shard a multiple of 8 elements, every buffer 16-byte aligned.
template <int CAP>
struct GatherTmaArgs {
  const uint16_t* src[CAP];
  uint16_t* full;
  int64_t numel;
  int64_t u8;     // numel rounded down to a multiple of 8: [0, u8) moves by TMA
  int64_t shard;  // a multiple of 8
  int32_t withhold;  // test hook: issue no loads, so every wait runs out
};

template <int CAP>
__global__ void __launch_bounds__(32, 1)
    zero3_unit_gather_tma_kernel(const __grid_constant__ GatherTmaArgs<CAP> a) {
  extern __shared__ __align__(1024) uint8_t ring[];
  __shared__ __align__(8) uint64_t bar[kSlots];
  const int lane = threadIdx.x;
  if (blockIdx.x == 0 && a.u8 + lane < a.numel && !a.withhold) {  // the last < 8 elements
    const int64_t e = a.u8 + lane;
    const int64_t r = e / a.shard;
    a.full[e] = a.src[r][e - r * a.shard];
  }
  const int64_t nchunks = (a.u8 + kChunk - 1) / kChunk;
  if (lane != 0 || blockIdx.x >= nchunks) return;
  for (int s = 0; s < kSlots; ++s) mbar_init(&bar[s], 1);
  mbar_init_fence();
  const int64_t mine = (nchunks - blockIdx.x + gridDim.x - 1) / gridDim.x;
  FlatLayout<GatherTmaArgs<CAP>> layout{a};
  ring_copy<kSlots>(layout, mine, ring, bar, a.withhold != 0, &g_gather_status);
}

template <int CAP>
bool launch_tma_cap(const GatherLaunch& L, cudaError_t* err) {
  const int64_t u8 = L.numel & ~static_cast<int64_t>(7);
  bool ok = u8 > 0 && L.shard % 8 == 0 && (reinterpret_cast<uintptr_t>(L.full) & 15u) == 0;
  for (int k = 0; k < L.world && ok; ++k)
    ok = (reinterpret_cast<uintptr_t>(L.shards[k]) & 15u) == 0;
  if (!ok) return false;
  static std::mutex mu;
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!configured[dev]) {
      if (cudaFuncSetAttribute(zero3_unit_gather_tma_kernel<CAP>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kRingBytes)) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
      }
      configured[dev] = true;
    }
  }
  int sms = 0;
  if (device_sm_count(&sms) != 0) return false;
  GatherTmaArgs<CAP> a;
  for (int k = 0; k < L.world; ++k) a.src[k] = L.shards[k];
  for (int k = L.world; k < CAP; ++k) a.src[k] = nullptr;
  a.full = L.full;
  a.numel = L.numel;
  a.u8 = u8;
  a.shard = L.shard;
  a.withhold = L.withhold;
  const int64_t nchunks = flat_chunks(u8);
  const int grid = static_cast<int>(nchunks < sms ? nchunks : sms);
  zero3_unit_gather_tma_kernel<CAP><<<grid, 32, kRingBytes, L.stream>>>(a);
  *err = cudaGetLastError();
  return true;
}

int gather_blocks_per_sm(const void* kernel) {
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

template <int CAP>
cudaError_t launch_cap(const GatherLaunch& L) {
  cudaError_t err = cudaSuccess;
  if (launch_tma_cap<CAP>(L, &err)) return err;
  GatherArgs<CAP> a;
  bool vec = (reinterpret_cast<uintptr_t>(L.full) % 16 == 0) && (L.world == 1 || L.shard % 8 == 0);
  for (int k = 0; k < L.world; ++k) {
    a.src[k] = L.shards[k];
    vec = vec && (reinterpret_cast<uintptr_t>(L.shards[k]) % 16 == 0);
  }
  for (int k = L.world; k < CAP; ++k) a.src[k] = nullptr;
  a.full = L.full;
  a.numel = L.numel;
  a.shard = L.shard;
  a.world = L.world;
  a.vec = vec ? 1 : 0;

  const void* kern = reinterpret_cast<const void*>(&zero3_unit_gather_kernel<CAP>);
  int sms = 0;
  if (device_sm_count(&sms) != 0) return cudaErrorNoDevice;
  const int64_t total = static_cast<int64_t>(sms) * gather_blocks_per_sm(kern);
  const int64_t per_shard_vec = (L.shard + 8 * kUnroll - 1) / (8 * kUnroll);
  int64_t bx = (per_shard_vec + kThreads - 1) / kThreads;
  int64_t cap = total / L.world;
  if (cap < 1) cap = 1;
  if (bx > cap) bx = cap;
  if (bx < 1) bx = 1;
  dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(L.world));
  zero3_unit_gather_kernel<CAP><<<grid, kThreads, 0, L.stream>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// FSDP2-style unit gather: every (tensor i, rank r) block of rows is one
// contiguous run in rank r's shard and one contiguous run of the unit, so the
// gather is ntensors*world block copies.  blockIdx.y strides over the blocks,
// blockIdx.x over a block's elements.

constexpr int kMaxTensors = 256;
// 8 vectors in flight per thread, at most 64 registers (4 blocks per SM):
// measured best for the row-block copies (a Llama-7B layer at N = 8 and 64).
constexpr int kRowsUnroll = 8;

template <int CAP>
struct GatherRowsArgs {
  const uint16_t* src[CAP];
  uint16_t* full;
  int32_t world, ntensors;
  int64_t rows[kMaxTensors], cols[kMaxTensors], per_rank[kMaxTensors];
  int64_t full_off[kMaxTensors], shard_off[kMaxTensors];
};

template <int CAP>
void fill_rows_args(const GatherRowsLaunch& L, GatherRowsArgs<CAP>* a) {
  for (int k = 0; k < L.world; ++k) a->src[k] = L.shards[k];
  for (int k = L.world; k < CAP; ++k) a->src[k] = nullptr;
  a->full = L.full;
  a->world = L.world;
  a->ntensors = L.ntensors;
  for (int i = 0; i < kMaxTensors; ++i) {
    const bool in = i < L.ntensors;
    a->rows[i] = in ? L.rows[i] : 0;
    a->cols[i] = in ? L.cols[i] : 0;
    a->per_rank[i] = in ? L.rows_per_rank[i] : 0;
    a->full_off[i] = in ? L.full_off[i] : 0;
    a->shard_off[i] = in ? L.shard_off[i] : 0;
  }
}

template <int CAP>
__global__ void __launch_bounds__(kThreads, 4)
    zero3_unit_gather_rows_kernel(const __grid_constant__ GatherRowsArgs<CAP> a) {
  const int64_t nseg = static_cast<int64_t>(a.ntensors) * a.world;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t seg = blockIdx.y; seg < nseg; seg += gridDim.y) {
    const int i = static_cast<int>(seg / a.world);
    const int r = static_cast<int>(seg - static_cast<int64_t>(i) * a.world);
    const int64_t r0 = static_cast<int64_t>(r) * a.per_rank[i];
    if (r0 >= a.rows[i]) continue;
    int64_t nrows = a.rows[i] - r0;
    if (nrows > a.per_rank[i]) nrows = a.per_rank[i];
    const int64_t len = nrows * a.cols[i];
    const uint16_t* __restrict__ src = a.src[r] + a.shard_off[i];
    uint16_t* __restrict__ dst = a.full + a.full_off[i] + r0 * a.cols[i];
    int64_t done = 0;
    if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u) == 0) {
      const int64_t nv = len / 8;
      const uint4* s4 = reinterpret_cast<const uint4*>(src);
      uint4* d4 = reinterpret_cast<uint4*>(dst);
      int64_t q = tid;
      for (; q + (kRowsUnroll - 1) * nthreads < nv; q += kRowsUnroll * nthreads) {
        uint4 x[kRowsUnroll];
#pragma unroll
        for (int u = 0; u < kRowsUnroll; ++u) x[u] = __ldcs(s4 + q + u * nthreads);
#pragma unroll
        for (int u = 0; u < kRowsUnroll; ++u) __stcs(d4 + q + u * nthreads, x[u]);
      }
      for (; q < nv; q += nthreads) __stcs(d4 + q, __ldcs(s4 + q));
      done = nv * 8;
    }
    for (int64_t j = done + tid; j < len; j += nthreads) dst[j] = __ldcs(src + j);
  }
}

// Row gather on the TMA engine: every row block (tensor i, rank r) is a run of
// nrows * cols elements at shard_off[i] in shard r and at
// full_off[i] + r * per_rank[i] * cols[i] in the unit.  With full_off[i] and
// per_rank[i] * cols[i] multiples of 8 (so shard_off[i] too) and every buffer
// 16-byte aligned, each run starts on a 16-byte boundary at both ends.  Every
// run of tensor i gets cps[i] = ceil(per_rank[i] * cols[i] / kChunk) chunk
// numbers (the short or empty runs of the last ranks leave some of theirs
// empty); chunk j belongs to the tensor i with prefix[i] <= j < prefix[i + 1].
template <int CAP>
struct RowsTmaArgs {
  GatherRowsArgs<CAP> g;
  int64_t cps[kMaxTensors];
  int64_t prefix[kMaxTensors + 1];
  int32_t withhold;  // test hook: issue no loads, so every wait runs out
};

// The CTA's chunks j = blockIdx.x + i * gridDim.x, walked as (tensor t, chunk k
// within the tensor's world * cps[t] chunks); tables in shared memory.
struct RowsTables {
  int64_t rows[kMaxTensors], cols[kMaxTensors], per_rank[kMaxTensors];
  int64_t full_off[kMaxTensors], shard_off[kMaxTensors], cps[kMaxTensors];
};

// Where a chunk held in a ring slot goes: one bulk store of `bytes` to `dst`.
struct Pending {
  uint16_t* dst;
  uint32_t bytes;
};

struct RowsLayout {
  const RowsTables& tb;
  const uint16_t* const* src;
  uint16_t* full;
  Pending* pending;  // per ring slot, filled when the chunk is loaded
  int32_t world, ntensors;
  int64_t t, k, stride;
  __device__ void skip() {  // move (t, k) past tensors whose chunks are used up
    while (t < ntensors && k >= world * tb.cps[t]) {
      k -= world * tb.cps[t];
      ++t;
    }
  }
  // chunk i is the next one of the walk: loads are issued in order
  __device__ void load(int64_t i, uint8_t* slot, uint64_t* bar) {
    const int64_t r = k / tb.cps[t];
    const int64_t e0 = (k - r * tb.cps[t]) * kChunk;
    const int64_t r0 = r * tb.per_rank[t];
    int64_t nrows = tb.rows[t] - r0;
    if (nrows > tb.per_rank[t]) nrows = tb.per_rank[t];
    if (nrows < 0) nrows = 0;
    const int64_t aligned = (nrows * tb.cols[t]) & ~static_cast<int64_t>(7);
    int64_t e1 = e0 + kChunk < aligned ? e0 + kChunk : aligned;
    if (e1 < e0) e1 = e0;
    const uint32_t bytes = static_cast<uint32_t>((e1 - e0) * 2);
    mbar_expect_tx(bar, bytes);
    if (bytes) bulk_load(slot, src[r] + tb.shard_off[t] + e0, bytes, bar);
    pending[i % kSlots] = Pending{full + tb.full_off[t] + r0 * tb.cols[t] + e0, bytes};
    k += stride;
    skip();
  }
  __device__ void store(int64_t i, const uint8_t* slot) const {
    const Pending& p = pending[i % kSlots];
    if (p.bytes) bulk_store(p.dst, slot, p.bytes);
  }
};

template <int CAP>
__global__ void __launch_bounds__(32, 1)
    zero3_unit_gather_rows_tma_kernel(const __grid_constant__ RowsTmaArgs<CAP> a) {
  extern __shared__ __align__(1024) uint8_t ring[];
  __shared__ __align__(8) uint64_t bar[kSlots];
  __shared__ Pending pending[kSlots];
  __shared__ RowsTables tb;
  __shared__ const uint16_t* src[CAP];
  const GatherRowsArgs<CAP>& g = a.g;
  const int lane = threadIdx.x;
  // the last (< 8) elements of every run, all lanes of all CTAs
  const int64_t nseg = static_cast<int64_t>(g.ntensors) * g.world;
  for (int64_t seg = static_cast<int64_t>(blockIdx.x) * 32 + lane; seg < nseg && !a.withhold;
       seg += static_cast<int64_t>(gridDim.x) * 32) {
    const int i = static_cast<int>(seg / g.world);
    const int64_t r = seg - static_cast<int64_t>(i) * g.world;
    const int64_t r0 = r * g.per_rank[i];
    int64_t nrows = g.rows[i] - r0;
    if (nrows > g.per_rank[i]) nrows = g.per_rank[i];
    if (nrows <= 0) continue;
    const int64_t len = nrows * g.cols[i];
    for (int64_t e = len & ~static_cast<int64_t>(7); e < len; ++e)
      g.full[g.full_off[i] + r0 * g.cols[i] + e] = g.src[r][g.shard_off[i] + e];
  }
  const int64_t nchunks = a.prefix[g.ntensors];
  if (blockIdx.x >= nchunks) return;
  for (int i = lane; i < g.ntensors; i += 32) {
    tb.rows[i] = g.rows[i];
    tb.cols[i] = g.cols[i];
    tb.per_rank[i] = g.per_rank[i];
    tb.full_off[i] = g.full_off[i];
    tb.shard_off[i] = g.shard_off[i];
    tb.cps[i] = a.cps[i];
  }
  for (int k = lane; k < g.world; k += 32) src[k] = g.src[k];
  __syncwarp();
  if (lane != 0) return;
  for (int s = 0; s < kSlots; ++s) mbar_init(&bar[s], 1);
  mbar_init_fence();
  const int64_t mine = (nchunks - blockIdx.x + gridDim.x - 1) / gridDim.x;
  RowsLayout layout{tb, src, g.full, pending, g.world, g.ntensors, 0, blockIdx.x, gridDim.x};
  layout.skip();
  ring_copy<kSlots>(layout, mine, ring, bar, a.withhold != 0, &g_gather_status);
}

template <int CAP>
bool launch_rows_tma(const GatherRowsLaunch& L, cudaError_t* err) {
  bool ok = (reinterpret_cast<uintptr_t>(L.full) & 15u) == 0;
  for (int k = 0; k < L.world && ok; ++k)
    ok = (reinterpret_cast<uintptr_t>(L.shards[k]) & 15u) == 0;
  for (int i = 0; i < L.ntensors && ok; ++i)
    ok = L.full_off[i] % 8 == 0 && L.shard_off[i] % 8 == 0 &&
         (L.rows_per_rank[i] * L.cols[i]) % 8 == 0;
  if (!ok) return false;
  static std::mutex mu;
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!configured[dev]) {
      if (cudaFuncSetAttribute(zero3_unit_gather_rows_tma_kernel<CAP>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kRingBytes)) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
      }
      configured[dev] = true;
    }
  }
  int sms = 0;
  if (device_sm_count(&sms) != 0) return false;
  RowsTmaArgs<CAP> a;
  fill_rows_args(L, &a.g);
  a.prefix[0] = 0;
  for (int i = 0; i < kMaxTensors; ++i) {
    a.cps[i] = i < L.ntensors ? (L.rows_per_rank[i] * L.cols[i] + kChunk - 1) / kChunk : 0;
    if (i < L.ntensors) a.prefix[i + 1] = a.prefix[i] + L.world * a.cps[i];
    else a.prefix[i + 1] = a.prefix[i];
  }
  a.withhold = L.withhold;
  const int64_t nchunks = a.prefix[L.ntensors];
  const int grid = static_cast<int>(nchunks < sms ? nchunks : sms);
  zero3_unit_gather_rows_tma_kernel<CAP><<<grid, 32, kRingBytes, L.stream>>>(a);
  *err = cudaGetLastError();
  return true;
}

template <int CAP>
cudaError_t launch_rows_cap(const GatherRowsLaunch& L) {
  cudaError_t err = cudaSuccess;
  if (launch_rows_tma<CAP>(L, &err)) return err;
  GatherRowsArgs<CAP> a;
  fill_rows_args(L, &a);
  int64_t biggest = 1;
  for (int i = 0; i < L.ntensors; ++i) {
    const int64_t blk = L.rows_per_rank[i] * L.cols[i];
    if (blk > biggest) biggest = blk;
  }

  const void* kern = reinterpret_cast<const void*>(&zero3_unit_gather_rows_kernel<CAP>);
  int sms = 0;
  if (device_sm_count(&sms) != 0) return cudaErrorNoDevice;
  const int64_t total = static_cast<int64_t>(sms) * gather_blocks_per_sm(kern);
  const int64_t nseg = static_cast<int64_t>(L.ntensors) * L.world;
  const int64_t gy = nseg < 65535 ? nseg : 65535;
  int64_t bx = (biggest / (8 * kRowsUnroll) + kThreads - 1) / kThreads;
  int64_t cap = total / gy;
  if (cap < 1) cap = 1;
  if (bx > cap) bx = cap;
  if (bx < 1) bx = 1;
  dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(gy));
  zero3_unit_gather_rows_kernel<CAP><<<grid, kThreads, 0, L.stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_unit_gather_rows(const GatherRowsLaunch& L) {
  (void)cudaGetLastError();
  if (L.world <= 8) return launch_rows_cap<8>(L);
  if (L.world <= 64) return launch_rows_cap<64>(L);
  return launch_rows_cap<1024>(L);
}

namespace {
__device__ int g_gather_status_taken;

// As take_step_status_kernel: one atomic exchange reads and clears the word.
__global__ void take_gather_status_kernel() {
  g_gather_status_taken = atomicExch(&g_gather_status, 0);
}
}  // namespace

int read_and_clear_gather_status(int* status) {
  take_gather_status_kernel<<<1, 1, 0, 0>>>();
  if (cudaGetLastError() != cudaSuccess) return -1;
  int v = 0;  // the copy is ordered after the kernel on the legacy default stream
  if (cudaMemcpyFromSymbol(&v, g_gather_status_taken, sizeof(int)) != cudaSuccess) return -1;
  *status = v;
  return 0;
}

cudaError_t launch_unit_gather(const GatherLaunch& L) {
  if (L.numel <= 0) return cudaSuccess;
  (void)cudaGetLastError();
  if (L.world <= 8) return launch_cap<8>(L);
  if (L.world <= 64) return launch_cap<64>(L);
  return launch_cap<1024>(L);
}

}  // namespace zeroadam
