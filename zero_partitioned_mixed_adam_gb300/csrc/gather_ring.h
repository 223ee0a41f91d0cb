// gather_ring.h -- the ZeRO-3 unit gather's copy on the TMA engine ("ZeRO and
// FSDP" -> "ZeRO-3 and FSDP": before a unit is used its complete parameters
// are all-gathered from the ranks' shards), shared by the gather kernels and
// the fused unit step.  Not installed; included by the kernel files of
// libzeroadam.so.
//
// A copy is cut into chunks of up to 8192 elements (16 KB) whose pieces all
// start on 16-byte boundaries and are multiples of 16 bytes long; the
// launchers check the layouts that guarantee it.  One thread moves its CTA's
// chunks through a ring of SLOTS slots in shared memory: bulk loads of a
// chunk's pieces into a slot, completing on the slot's mbarrier, then one bulk
// store of the slot, committed as a bulk async-group.  Loads run SLOTS - 1
// chunks ahead; a slot is reloaded once the store that read it has finished
// reading.
//
// Every wait is bounded by the global timer; a wait that gives up writes a
// nonzero value to the caller's status word, waits (bounded) for the loads
// already issued and for its stores, and stops.
#pragma once

#include <cstdint>

#include "tma_ops.h"

namespace zeroadam {

constexpr int kChunk = 8192;  // elements per chunk
constexpr int kSlots = 4;     // ring of 4 x 16 KB (the gather kernels)
constexpr int64_t kSlotBytes = static_cast<int64_t>(kChunk) * 2;
constexpr size_t kRingBytes = static_cast<size_t>(kSlots) * kSlotBytes;

// One thread moves its CTA's `mine` chunks (chunk i of the CTA is chunk
// blockIdx.x + i * gridDim.x of the copy) through the ring.  layout.load(i,
// slot, bar) issues the bulk loads of the CTA's chunk i into `slot` and arms
// `bar` with their byte count (zero bytes: the arrive alone completes the
// phase); it is called for i = 0, 1, 2, ... in order.  layout.store(i, slot)
// issues chunk i's bulk store, if it has any bytes.
template <int SLOTS, class Layout>
__device__ void ring_copy(Layout& layout, int64_t mine, uint8_t* ring, uint64_t* bar,
                          bool withhold, int* status) {
  static_assert(SLOTS >= 2, "a slot is reloaded only after its store has read it");
  auto load = [&](int64_t i) {
    if (!withhold) layout.load(i, ring + (i % SLOTS) * kSlotBytes, &bar[i % SLOTS]);
  };
  int64_t loaded = mine < SLOTS - 1 ? mine : SLOTS - 1;
  for (int64_t i = 0; i < loaded; ++i) load(i);
  for (int64_t i = 0; i < mine; ++i) {
    const int s = static_cast<int>(i % SLOTS);
    if (!mbar_wait(&bar[s], static_cast<uint32_t>((i / SLOTS) & 1))) {
      atomicExch(status, 1);
      for (int64_t j = i; j < loaded && !withhold; ++j)  // issued loads land first
        mbar_wait(&bar[j % SLOTS], static_cast<uint32_t>((j / SLOTS) & 1));
      break;
    }
    fence_async_shared();
    layout.store(i, ring + s * kSlotBytes);
    bulk_commit();
    if (i + SLOTS - 1 < mine) {
      bulk_wait_read<1>();  // the store of chunk i - 1 has read slot (i - 1) % SLOTS
      load(i + SLOTS - 1);
      ++loaded;
    }
  }
  bulk_wait_all();
}

// Flat gather (zero3_unit_gather's layout): full[r*shard + j] = src[r][j].
// Args holds src[] (the shards), full, u8 (numel rounded down to a multiple of
// 8: [0, u8) moves by TMA) and shard (a multiple of 8, so every piece starts
// on a 16-byte boundary).  The CTA's chunk i covers [e0, e1), e0 =
// (blockIdx.x + i * gridDim.x) * kChunk; a chunk is one piece per shard it
// touches.
template <class Args>
struct FlatLayout {
  const Args& a;
  __device__ void range(int64_t i, int64_t* e0, int64_t* e1) const {
    *e0 = (blockIdx.x + i * static_cast<int64_t>(gridDim.x)) * kChunk;
    *e1 = *e0 + kChunk < a.u8 ? *e0 + kChunk : a.u8;
  }
  __device__ void load(int64_t i, uint8_t* slot, uint64_t* bar) const {
    int64_t e0, e1;
    range(i, &e0, &e1);
    mbar_expect_tx(bar, static_cast<uint32_t>((e1 - e0) * 2));
    for (int64_t e = e0; e < e1;) {
      const int64_t r = e / a.shard;
      const int64_t pe = (r + 1) * a.shard < e1 ? (r + 1) * a.shard : e1;
      bulk_load(slot + (e - e0) * 2, a.src[r] + (e - r * a.shard),
                static_cast<uint32_t>((pe - e) * 2), bar);
      e = pe;
    }
  }
  __device__ void store(int64_t i, const uint8_t* slot) const {
    int64_t e0, e1;
    range(i, &e0, &e1);
    bulk_store(a.full + e0, slot, static_cast<uint32_t>((e1 - e0) * 2));
  }
};

// Chunks of a flat gather of u8 elements.
__host__ __device__ constexpr int64_t flat_chunks(int64_t u8) { return (u8 + kChunk - 1) / kChunk; }

}  // namespace zeroadam
