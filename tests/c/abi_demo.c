/*
 * abi_demo.c -- a plain C11 user of libzeroadam.so through include/zeroadam.h.
 *
 *   abi_demo plan   : host-only checks (no GPU needed): the planner and the
 *                     status codes of bad arguments.
 *   abi_demo step   : one all-ranks step on the GPU with cudaMalloc'd
 *                     buffers, zero gradients and m = v = 0, where Adam leaves
 *                     the master weights unchanged and the bf16 parameters are
 *                     their round-to-nearest-even cast.
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

int main(int argc, char** argv) {
  if (argc > 1 && strcmp(argv[1], "step") == 0) return step_check();
  return plan_checks();
}
