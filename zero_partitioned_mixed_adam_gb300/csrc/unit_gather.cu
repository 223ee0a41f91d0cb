// unit_gather.cu -- ZeRO-3 unit all-gather on sm_103a ("ZeRO and FSDP" ->
// "ZeRO-3 and FSDP": before a unit is used its complete parameters are
// all-gathered from the ranks' shards).  With the ranks emulated in one
// GPU's memory the gather is a copy of N bf16 shards into one unit buffer:
//   full[r*shard + j] = shard_r[j],  r*shard + j < numel.
// It moves 4 bytes per unit element (2 read, 2 written) and is bound by HBM
// bandwidth, or for small units by launch latency.
#include <mutex>
#include <unordered_map>

#include "internal.h"

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

template <int CAP>
cudaError_t launch_rows_cap(const GatherRowsLaunch& L) {
  GatherRowsArgs<CAP> a;
  for (int k = 0; k < L.world; ++k) a.src[k] = L.shards[k];
  for (int k = L.world; k < CAP; ++k) a.src[k] = nullptr;
  a.full = L.full;
  a.world = L.world;
  a.ntensors = L.ntensors;
  int64_t biggest = 1;
  for (int i = 0; i < L.ntensors; ++i) {
    a.rows[i] = L.rows[i];
    a.cols[i] = L.cols[i];
    a.per_rank[i] = L.rows_per_rank[i];
    a.full_off[i] = L.full_off[i];
    a.shard_off[i] = L.shard_off[i];
    const int64_t blk = L.rows_per_rank[i] * L.cols[i];
    if (blk > biggest) biggest = blk;
  }
  for (int i = L.ntensors; i < kMaxTensors; ++i)
    a.rows[i] = a.cols[i] = a.per_rank[i] = a.full_off[i] = a.shard_off[i] = 0;

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

cudaError_t launch_unit_gather(const GatherLaunch& L) {
  if (L.numel <= 0) return cudaSuccess;
  (void)cudaGetLastError();
  if (L.world <= 8) return launch_cap<8>(L);
  if (L.world <= 64) return launch_cap<64>(L);
  return launch_cap<1024>(L);
}

}  // namespace zeroadam
