// internal.h -- declarations shared by the C-ABI layer and the kernel files of
// libzeroadam.so.  Not installed; the public interface is include/zeroadam.h.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace zeroadam {

// The step's binary32 scalars.  Each is formed in double on the host and
// rounded to binary32 once (the page's step mixes Python floats, i.e. doubles,
// into fp32 tensor expressions).
struct AdamScalars {
  float b1, omb1;    // beta1, 1 - beta1
  float b2, omb2;    // beta2, 1 - beta2
  float bc1, bc2;    // 1 - beta1^t, 1 - beta2^t
  float lr, eps;
  float world;       // N as binary32
  float inv_world;   // 1/N, exact when N is a power of two
  int32_t pow2_world;  // N is a power of two: g/N == g*(1/N) exactly
};

// One launch of the fused step over a contiguous range of n flat elements.
// Every pointer already points at the range's first element.
struct StepLaunch {
  const void* const* grads;  // host array of `world` device pointers (bf16, or fp32 if grad_f32)
  int32_t world;
  int32_t grad_f32;  // gradients are fp32 (else bf16)
  int32_t acc_bf16;  // the running sum over ranks is rounded to bf16 after every addition
  float* master;
  float* m;
  float* v;
  uint16_t* param;
  int64_t n;
  AdamScalars s;
  cudaStream_t stream;
  int32_t withhold;  // test hook for the TMA-staged kernels (zero_test_withhold_copies)
};

// One launch of the ZeRO-3 unit gather.
struct GatherLaunch {
  const uint16_t* const* shards;  // host array of `world` device pointers (bf16)
  int32_t world;
  uint16_t* full;
  int64_t numel;
  int64_t shard;
  cudaStream_t stream;
  int32_t withhold;  // test hook for the TMA gather kernel (zero_test_withhold_copies)
};

// One launch of the FSDP2-style (dim-0 row-sharded) unit gather.  Offsets are
// in elements; rows_per_rank = ceil(rows / world).
struct GatherRowsLaunch {
  const uint16_t* const* shards;
  int32_t world;
  int32_t ntensors;
  const int64_t* rows;
  const int64_t* cols;
  const int64_t* rows_per_rank;
  const int64_t* full_off;
  const int64_t* shard_off;
  uint16_t* full;
  cudaStream_t stream;
  int32_t withhold;  // test hook for the TMA row gather kernel (zero_test_withhold_copies)
};

// Streaming-multiprocessor count of the current device (cached per device).
int device_sm_count(int* sms);

cudaError_t launch_adam_step(const StepLaunch& L);
// Status word of the step kernels' bounded waits on the current device (0 =
// every wait completed); read and cleared.  Returns -1 if CUDA fails.
int read_and_clear_step_status(int* status);
cudaError_t launch_unit_gather(const GatherLaunch& L);
// Status word of the TMA gather kernel's bounded waits; as above.
int read_and_clear_gather_status(int* status);
cudaError_t launch_unit_gather_rows(const GatherRowsLaunch& L);
// The unit gather GL and the step L in one launch where both parts can run on
// the TMA engine, else the two launches in that order; the same results.
cudaError_t launch_unit_step(const GatherLaunch& GL, const StepLaunch& L);

}  // namespace zeroadam
