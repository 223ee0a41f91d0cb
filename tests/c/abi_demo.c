/*
 * abi_demo.c -- a plain C11 user of libzeroadam.so through include/zeroadam.h.
 *
 *   abi_demo plan   : host-only checks (no GPU needed): the planner and the
 *                     status codes of bad arguments.
 *   abi_demo step   : one all-ranks step on the GPU with cudaMalloc'd
 *                     buffers, zero gradients and m = v = 0, where Adam leaves
 *                     the master weights unchanged and the bf16 parameters are
 *                     their round-to-nearest-even cast.
 *   abi_demo unit   : one ZeRO-3 unit step (gather + one rank's step in one
 *                     call) on 8 ranks' shards: the gathered unit is the
 *                     shards back to back, bit for bit, and the rank's step
 *                     under a zero gradient behaves as above; the device
 *                     status afterwards is ZERO_OK.
 * Exit status 0 on success.
 */
#include <cuda_runtime_api.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "zeroadam.h"

static int fail(const char* what) {
  fprintf(stderr, "abi_demo: %s\n", what);
  return 1;
}

static int plan_checks(void) {
  zero_plan_t p;
  if (zero_plan(1000003, 4, &p) != ZERO_OK) return fail("zero_plan");
  if (p.shard != 250001 || p.pad != 1 || p.padded != 1000004) return fail("layout");
  if (p.bytes_z2 != 2u * 1000003u + 14u * 250001u) return fail("ZeRO-2 bytes");
  if (zero_plan(0, 4, &p) != ZERO_E_NUMEL) return fail("numel 0 accepted");
  if (zero_plan(10, 0, &p) != ZERO_E_WORLD) return fail("world 0 accepted");
  if (zero_adam_step(NULL, -1, NULL, 0, NULL, NULL, NULL, NULL, 0, 1e-3, .9, .999, 1e-8, 1,
                     NULL) != ZERO_E_NULLPTR)
    return fail("NULL plan accepted");
  zero_plan(100, 2, &p);
  const void* g[2] = {(void*)0x10000, (void*)0x20000};
  if (zero_adam_step(&p, ZERO_ALL_RANKS, g, ZERO_GRAD_FULL, (float*)0x30000, (float*)0x40000,
                     (float*)0x50000, (void*)0x60000, ZERO_PARAM_FULL, 1e-3, .9, .999, 1e-8, 0,
                     NULL) != ZERO_E_STEP)
    return fail("t = 0 accepted");
  printf("plan ok: shard %lld pad %lld, Z2 %.0f B/card; %s\n", (long long)250001, 1LL,
         (double)(2u * 1000003u + 14u * 250001u), zero_strerror(ZERO_E_STEP));
  return 0;
}

static uint16_t bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  const uint32_t lsb = (u >> 16) & 1u;
  return (uint16_t)((u + 0x7fffu + lsb) >> 16);
}

static int step_check(void) {
  const int64_t numel = 100003;
  const int32_t world = 4;
  zero_plan_t p;
  if (zero_plan(numel, world, &p) != ZERO_OK) return fail("zero_plan");
  const size_t P = (size_t)p.padded;
  float* hw = (float*)malloc(P * sizeof(float));
  for (size_t i = 0; i < P; ++i) hw[i] = i < (size_t)numel ? 0.01f * (float)((i % 97) - 48) : 0.f;
  void* g[4];
  float *w, *m, *v;
  uint16_t* par;
  for (int k = 0; k < world; ++k) {
    if (cudaMalloc(&g[k], P * 2) != cudaSuccess) return fail("cudaMalloc");
    cudaMemset(g[k], 0, P * 2);
  }
  cudaMalloc((void**)&w, P * 4);
  cudaMalloc((void**)&m, P * 4);
  cudaMalloc((void**)&v, P * 4);
  cudaMalloc((void**)&par, (size_t)numel * 2);
  cudaMemcpy(w, hw, P * 4, cudaMemcpyHostToDevice);
  cudaMemset(m, 0, P * 4);
  cudaMemset(v, 0, P * 4);
  const int rc = zero_adam_step(&p, ZERO_ALL_RANKS, (const void* const*)g, ZERO_GRAD_FULL, w, m,
                                v, par, ZERO_PARAM_FULL, 1e-3, 0.9, 0.999, 1e-8, 1, NULL);
  if (rc != ZERO_OK) return fail(zero_strerror(rc));
  if (cudaDeviceSynchronize() != cudaSuccess) return fail("kernel");
  float* w2 = (float*)malloc(P * 4);
  uint16_t* p2 = (uint16_t*)malloc((size_t)numel * 2);
  cudaMemcpy(w2, w, P * 4, cudaMemcpyDeviceToHost);
  cudaMemcpy(p2, par, (size_t)numel * 2, cudaMemcpyDeviceToHost);
  for (int64_t i = 0; i < numel; ++i) {
    if (memcmp(&w2[i], &hw[i], 4) != 0) return fail("master changed under a zero gradient");
    if (p2[i] != bf16_rne(hw[i])) return fail("bf16 parameter is not the cast of the master");
  }
  printf("step ok: %lld elements, zero gradient leaves the master, params = bf16(master)\n",
         (long long)numel);
  return 0;
}

static int unit_check(void) {
  const int64_t numel = 1000000;
  const int32_t world = 8, rank = 5;
  zero_plan_t p;
  if (zero_plan(numel, world, &p) != ZERO_OK) return fail("zero_plan");
  const size_t S = (size_t)p.shard;
  uint16_t* hs = (uint16_t*)malloc(S * 2);
  float* hw = (float*)malloc(S * 4);
  void* shards[8];
  void* grads[8];
  for (int r = 0; r < world; ++r) {
    for (size_t j = 0; j < S; ++j) hs[j] = (uint16_t)(0x3c00u + ((uint32_t)r * 977u + (uint32_t)j) % 4093u);
    if (cudaMalloc(&shards[r], S * 2) != cudaSuccess) return fail("cudaMalloc");
    cudaMemcpy(shards[r], hs, S * 2, cudaMemcpyHostToDevice);
    if (cudaMalloc(&grads[r], S * 2) != cudaSuccess) return fail("cudaMalloc");
    cudaMemset(grads[r], 0, S * 2);
  }
  for (size_t j = 0; j < S; ++j) hw[j] = 0.003f * (float)((int)(j % 211) - 105);
  void* full;
  float *w, *m, *v;
  uint16_t* par;
  cudaMalloc(&full, (size_t)numel * 2);
  cudaMalloc((void**)&w, S * 4);
  cudaMalloc((void**)&m, S * 4);
  cudaMalloc((void**)&v, S * 4);
  cudaMalloc((void**)&par, S * 2);
  cudaMemcpy(w, hw, S * 4, cudaMemcpyHostToDevice);
  cudaMemset(m, 0, S * 4);
  cudaMemset(v, 0, S * 4);
  cudaMemset(full, 0xff, (size_t)numel * 2);
  const int rc = zero3_unit_step(&p, rank, (const void* const*)shards, full,
                                 (const void* const*)grads, ZERO_GRAD_SHARD, w, m, v, par,
                                 ZERO_PARAM_SHARD, 1e-3, 0.9, 0.999, 1e-8, 1, NULL);
  if (rc != ZERO_OK) return fail(zero_strerror(rc));
  const int st = zero_device_status();
  if (st != ZERO_OK) return fail(zero_strerror(st));
  uint16_t* hf = (uint16_t*)malloc((size_t)numel * 2);
  float* w2 = (float*)malloc(S * 4);
  uint16_t* p2 = (uint16_t*)malloc(S * 2);
  cudaMemcpy(hf, full, (size_t)numel * 2, cudaMemcpyDeviceToHost);
  cudaMemcpy(w2, w, S * 4, cudaMemcpyDeviceToHost);
  cudaMemcpy(p2, par, S * 2, cudaMemcpyDeviceToHost);
  for (int64_t i = 0; i < numel; ++i) {
    const uint32_t r = (uint32_t)(i / (int64_t)S), j = (uint32_t)(i % (int64_t)S);
    if (hf[i] != (uint16_t)(0x3c00u + (r * 977u + j) % 4093u)) return fail("gathered unit differs");
  }
  for (size_t j = 0; j < S; ++j) {
    if (memcmp(&w2[j], &hw[j], 4) != 0) return fail("master changed under a zero gradient");
    if (p2[j] != bf16_rne(hw[j])) return fail("bf16 shard is not the cast of the master");
  }
  printf("unit ok: %lld-element unit gathered from %d shards, rank %d stepped, status ok\n",
         (long long)numel, world, rank);
  return 0;
}

int main(int argc, char** argv) {
  if (argc > 1 && strcmp(argv[1], "step") == 0) return step_check();
  if (argc > 1 && strcmp(argv[1], "unit") == 0) return unit_check();
  return plan_checks();
}
