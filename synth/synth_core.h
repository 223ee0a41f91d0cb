/*
 * synth_core.h -- seeded, counter-based synthetic inputs for the ZeRO Adam step.
 *
 * This module produces the INPUTS only (gradients, master weights, parameter
 * shards).  It holds none of the optimizer's arithmetic: no reduction over
 * ranks, no Adam, no fp32->bf16 round-to-nearest cast.  bf16 values are made
 * by truncating an fp32 draw to its top 16 bits, which is a valid bf16 sample
 * of (almost) the same distribution and needs no rounding code.
 *
 * The same header is compiled twice: by gcc for the host generator and by nvcc
 * for the device generator.  Every floating-point step is one IEEE binary32
 * operation with round-to-nearest-even and no contraction into FMA (device:
 * the __f*_rn intrinsics; host: -ffp-contract=off), and the only non-basic
 * operation, the natural log, is computed here from its series with +,-,*,/.
 * Hence the host and the device produce bit-identical values.
 *
 * Generator (published definitions):
 *   mix64     : the SplitMix64 output finaliser (Steele, Lea, Flood,
 *               "Fast splittable pseudorandom number generators", OOPSLA 2014;
 *               constants of Stafford's "Mix13").
 *   key       : mix64 chained over (seed, stream, rank, step).
 *   word(k,c) : mix64(k + GAMMA*(c+1)) -- a counter-based stream; element i of a
 *               buffer uses counters derived from its GLOBAL index, so any
 *               window of a buffer can be regenerated on its own.
 *   uniform   : top 24 bits of a word times 2^-24, in [0,1).
 *   normal    : Marsaglia's polar method (Marsaglia & Bray, SIAM Review 1964),
 *               at most 32 attempts, each with its own two counters.
 *   ln(s)     : s = f*2^e with f in [sqrt(1/2), sqrt(2)); ln s = e*ln2 +
 *               2*atanh((f-1)/(f+1)), atanh by its Taylor series to t^9.
 *   Student-t(3) = z0 / sqrt((z1^2+z2^2+z3^2)/3).
 */
#ifndef SYNTH_CORE_H
#define SYNTH_CORE_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYN_HD __host__ __device__ __forceinline__
#else
#define SYN_HD static inline
#endif

#if defined(__CUDA_ARCH__)
#define SYN_ADD(a, b) __fadd_rn((a), (b))
#define SYN_SUB(a, b) __fsub_rn((a), (b))
#define SYN_MUL(a, b) __fmul_rn((a), (b))
#define SYN_DIV(a, b) __fdiv_rn((a), (b))
#define SYN_SQRT(a) __fsqrt_rn(a)
#else
#include <math.h>
#define SYN_ADD(a, b) ((float)((a) + (b)))
#define SYN_SUB(a, b) ((float)((a) - (b)))
#define SYN_MUL(a, b) ((float)((a) * (b)))
#define SYN_DIV(a, b) ((float)((a) / (b)))
#define SYN_SQRT(a) sqrtf(a)
#endif

#define SYN_GAMMA 0x9E3779B97F4A7C15ull

/* Distribution codes. */
enum { SYNTH_NORMAL = 0, SYNTH_STUDENT_T3 = 1, SYNTH_CONSTANT = 2 };

/* Output element type. */
enum { SYNTH_OUT_F32 = 0, SYNTH_OUT_BF16 = 1 };

/*
 * One buffer's recipe.  value(i) = sigma * X_i, where X_i is N(0,1) or
 * Student-t(3); then, with probability zero_thr/2^64 (shared by all ranks: the
 * mask key leaves the rank out), value = 0; else with probability
 * outlier_thr/2^64 (per rank), value = +-outlier_value.  SYNTH_CONSTANT gives
 * value(i) = sigma for every i.
 */
typedef struct {
  uint64_t seed;
  uint32_t stream, rank, step, dist;
  float sigma;
  float outlier_value;
  uint64_t zero_thr;     /* 0 = no zero mask */
  uint64_t outlier_thr;  /* 0 = no outliers */
} synth_spec_t;

SYN_HD uint64_t syn_mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z;
}

SYN_HD uint64_t syn_key(uint64_t seed, uint32_t stream, uint32_t rank, uint32_t step) {
  uint64_t k = syn_mix64(seed + SYN_GAMMA);
  k = syn_mix64(k + SYN_GAMMA * ((uint64_t)stream + 1));
  k = syn_mix64(k + SYN_GAMMA * ((uint64_t)rank + 1));
  k = syn_mix64(k + SYN_GAMMA * ((uint64_t)step + 1));
  return k;
}

SYN_HD uint64_t syn_word(uint64_t key, uint64_t counter) {
  return syn_mix64(key + SYN_GAMMA * (counter + 1));
}

SYN_HD float syn_uniform(uint64_t w) {
  /* (w >> 40) < 2^24 is exact in binary32; the scale is a power of two. */
  return SYN_MUL((float)(uint32_t)(w >> 40), 5.9604644775390625e-08f);
}

SYN_HD uint32_t syn_f2u(float x) {
  union { float f; uint32_t u; } c;
  c.f = x;
  return c.u;
}

SYN_HD float syn_u2f(uint32_t u) {
  union { float f; uint32_t u; } c;
  c.u = u;
  return c.f;
}

/* Natural log of a positive normal binary32 s, from the atanh series. */
SYN_HD float syn_ln(float s) {
  uint32_t b = syn_f2u(s);
  int e = (int)((b >> 23) & 0xffu) - 127;
  float f = syn_u2f((b & 0x007fffffu) | 0x3f800000u); /* f in [1,2) */
  if (f > 1.41421353816986083984375f) {                 /* binary32 below sqrt(2) */
    f = SYN_MUL(f, 0.5f);
    e += 1;
  }
  const float t = SYN_DIV(SYN_SUB(f, 1.0f), SYN_ADD(f, 1.0f));
  const float t2 = SYN_MUL(t, t);
  float p = SYN_DIV(1.0f, 9.0f);
  p = SYN_ADD(SYN_DIV(1.0f, 7.0f), SYN_MUL(t2, p));
  p = SYN_ADD(SYN_DIV(1.0f, 5.0f), SYN_MUL(t2, p));
  p = SYN_ADD(SYN_DIV(1.0f, 3.0f), SYN_MUL(t2, p));
  p = SYN_ADD(1.0f, SYN_MUL(t2, p));
  const float atanh2 = SYN_MUL(2.0f, SYN_MUL(t, p));
  const float ln2 = 0.693147182464599609375f; /* binary32 nearest ln 2 */
  return SYN_ADD(SYN_MUL((float)e, ln2), atanh2);
}

/* Standard normal number n (0..3) of element i under key k. */
SYN_HD float syn_normal(uint64_t key, uint64_t i, uint32_t n) {
  const uint64_t base = (i * 4u + n) * 64u;
  for (uint32_t a = 0; a < 32u; ++a) {
    const float x = SYN_SUB(SYN_MUL(2.0f, syn_uniform(syn_word(key, base + 2u * a))), 1.0f);
    const float y = SYN_SUB(SYN_MUL(2.0f, syn_uniform(syn_word(key, base + 2u * a + 1u))), 1.0f);
    const float s = SYN_ADD(SYN_MUL(x, x), SYN_MUL(y, y));
    if (s < 1.0f && s > 0.0f) {
      const float r = SYN_SQRT(SYN_DIV(SYN_MUL(-2.0f, syn_ln(s)), s));
      return SYN_MUL(x, r);
    }
  }
  return 0.0f;
}

/* The fp32 value of element i (global index) of the buffer described by sp. */
SYN_HD float syn_value(const synth_spec_t* sp, uint64_t i) {
  if (sp->dist == SYNTH_CONSTANT) return sp->sigma;
  if (sp->zero_thr != 0u) {
    const uint64_t kz = syn_key(sp->seed, sp->stream + 0x10000u, 0u, sp->step);
    if (syn_word(kz, i) < sp->zero_thr) return 0.0f;
  }
  const uint64_t k = syn_key(sp->seed, sp->stream, sp->rank, sp->step);
  if (sp->outlier_thr != 0u) {
    const uint64_t ko = syn_key(sp->seed, sp->stream + 0x20000u, sp->rank, sp->step);
    const uint64_t w = syn_word(ko, i);
    if (w < sp->outlier_thr) return (w & 1u) ? -sp->outlier_value : sp->outlier_value;
  }
  float x = syn_normal(k, i, 0u);
  if (sp->dist == SYNTH_STUDENT_T3) {
    const float z1 = syn_normal(k, i, 1u);
    const float z2 = syn_normal(k, i, 2u);
    const float z3 = syn_normal(k, i, 3u);
    const float chi = SYN_ADD(SYN_ADD(SYN_MUL(z1, z1), SYN_MUL(z2, z2)), SYN_MUL(z3, z3));
    const float den = SYN_SQRT(SYN_DIV(chi, 3.0f));
    x = (den > 0.0f) ? SYN_DIV(x, den) : 0.0f;
  }
  return SYN_MUL(sp->sigma, x);
}

/* bf16 bits of a draw: the top half of the binary32 (truncation, not a cast). */
SYN_HD uint16_t syn_trunc_bf16(float x) { return (uint16_t)(syn_f2u(x) >> 16); }

#endif /* SYNTH_CORE_H */
