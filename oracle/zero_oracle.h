/*
 * zero_oracle.h -- the oracle's own declarations (test infrastructure only;
 * shares nothing with the CUDA library's header).
 */
#ifndef ZERO_ORACLE_H
#define ZERO_ORACLE_H

#include <stdint.h>

#define ORACLE_MAX_WORLD 1024

typedef struct {
  int64_t numel, world, shard, pad, padded;
  uint64_t bytes_dp, bytes_z1, bytes_z2, bytes_z3;
  double formula_dp, formula_z1, formula_z2, formula_z3;
  uint64_t state_bytes_rank;
  double comm_dp, comm_z1, comm_z2, comm_z3;
} oracle_plan_t;

typedef struct {
  float b1, omb1, b2, omb2, bc1, bc2, lr, eps, world;
} oracle_scalars_t;

int oracle_plan(int64_t numel, int32_t world, oracle_plan_t* out);
float oracle_bf16_to_f32(uint16_t h);
uint16_t oracle_f32_to_bf16(float f);
void oracle_scalars(double lr, double beta1, double beta2, double eps, int64_t t, int32_t world,
                    oracle_scalars_t* s);
int oracle_zero_step(const oracle_plan_t* plan, int32_t rank, int64_t i0, int64_t i1,
                     const uint16_t* const* grads, int64_t grad_base, float* master, float* m,
                     float* v, int64_t state_base, uint16_t* param, int64_t param_base, double lr,
                     double beta1, double beta2, double eps, int64_t t);
int oracle_zero_step_ex(const oracle_plan_t* plan, int32_t rank, int64_t i0, int64_t i1,
                        const void* const* grads, int64_t grad_base, int grad_f32, int acc_bf16,
                        float* master, float* m, float* v, int64_t state_base, uint16_t* param,
                        int64_t param_base, double lr, double beta1, double beta2, double eps,
                        int64_t t);
int oracle_dp_step(int64_t numel, int32_t world, const uint16_t* const* grads, float* master,
                   float* m, float* v, uint16_t* param, double lr, double beta1, double beta2,
                   double eps, int64_t t);
int oracle_unit_gather(int64_t unit_numel, int32_t world, const uint16_t* const* shards,
                       uint16_t* full);
int oracle_unit_gather_rows(int32_t ntensors, const int64_t* rows, const int64_t* cols,
                            int32_t world, const uint16_t* const* shards, uint16_t* full);
void oracle_f32_to_bf16_array(const float* x, uint16_t* out, int64_t n);

#endif
