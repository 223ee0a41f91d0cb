/*
 * synth_dev.cu -- device generator of the seeded synthetic inputs.
 * Bit-identical to synth_host.c: both evaluate synth_core.h, whose device
 * arithmetic is spelled with the round-to-nearest intrinsics.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include "synth_core.h"

template <int KIND>
__global__ void synth_fill_kernel(synth_spec_t s, int64_t offset, int64_t n, void* out) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float x = syn_value(&s, (uint64_t)(offset + i));
    if (KIND == SYNTH_OUT_F32)
      static_cast<float*>(out)[i] = x;
    else
      static_cast<uint16_t*>(out)[i] = syn_trunc_bf16(x);
  }
}

extern "C" {

/* Device counterpart of synth_fill_host; out is a device pointer, stream a
   cudaStream_t (NULL = legacy default stream).  Returns 0, -1 on a bad
   argument, -2 if the launch failed. */
int synth_fill_dev(const synth_spec_t* sp, int64_t offset, int64_t n, void* out, int out_kind,
                   void* stream) {
  if (sp == nullptr || (out == nullptr && n > 0) || n < 0 || offset < 0) return -1;
  if (n == 0) return 0;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 1;
  const int threads = 256;
  int64_t blocks = (n + threads - 1) / threads;
  const int64_t cap = (int64_t)sms * 16;
  if (blocks > cap) blocks = cap;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (out_kind == SYNTH_OUT_F32)
    synth_fill_kernel<SYNTH_OUT_F32><<<(unsigned)blocks, threads, 0, st>>>(*sp, offset, n, out);
  else if (out_kind == SYNTH_OUT_BF16)
    synth_fill_kernel<SYNTH_OUT_BF16><<<(unsigned)blocks, threads, 0, st>>>(*sp, offset, n, out);
  else
    return -1;
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

}  // extern "C"
