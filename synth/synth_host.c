/*
 * synth_host.c -- host (CPU) generator of the seeded synthetic inputs.
 * Bit-identical to synth_dev.cu: both evaluate synth_core.h.
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fopenmp -shared -fPIC.
 */
#include <stddef.h>
#include <stdint.h>

#include "synth_core.h"

/* Fill out[0..n) with elements offset..offset+n-1 of the buffer sp describes.
   out_kind: SYNTH_OUT_F32 (float*) or SYNTH_OUT_BF16 (uint16_t* bf16 bits).
   Returns 0, or -1 on a bad argument. */
int synth_fill_host(const synth_spec_t* sp, int64_t offset, int64_t n, void* out, int out_kind) {
  if (sp == NULL || (out == NULL && n > 0) || n < 0 || offset < 0) return -1;
  if (out_kind != SYNTH_OUT_F32 && out_kind != SYNTH_OUT_BF16) return -1;
  const synth_spec_t s = *sp;
  if (out_kind == SYNTH_OUT_F32) {
    float* o = (float*)out;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) o[i] = syn_value(&s, (uint64_t)(offset + i));
  } else {
    uint16_t* o = (uint16_t*)out;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) o[i] = syn_trunc_bf16(syn_value(&s, (uint64_t)(offset + i)));
  }
  return 0;
}

/* Exposed for the generator's own tests. */
float synth_ln_host(float s) { return syn_ln(s); }
uint64_t synth_mix64_host(uint64_t z) { return syn_mix64(z); }
