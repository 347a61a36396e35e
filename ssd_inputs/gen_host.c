/*
 * Host generator of the seeded synthetic inputs (definition in gen_def.h).
 * Used by the CPU oracle and by tests; built as libssd_inputs_host.so with
 * gcc + OpenMP.  No CUDA, no part of the decoding method.
 */
#include <math.h>
#include <stdint.h>

#include "gen_def.h"

static uint16_t value_bits(uint64_t key, uint64_t i, double mean, double sigma, int fp16) {
  const double two_pi = 6.283185307179586476925286766559;
  uint64_t r1 = ssdi_mix(key + 2 * i);
  uint64_t r2 = ssdi_mix(key + 2 * i + 1);
  double z = sqrt(-2.0 * log(ssdi_u1(r1))) * cos(two_pi * ssdi_u2(r2));
  float f = (float)(mean + sigma * z);
  if (fp16) {
    union { _Float16 h; uint16_t u; } v;
    v.h = (_Float16)f;
    return v.u;
  }
  return ssdi_f32_to_bf16_bits(f);
}

/* out[k] = value of element (offset + k) of tensor `tensor_id`, k < n:
   round16((float)(mean + sigma * z)). */
void ssd_inputs_fill_host(uint16_t* out, uint64_t n, uint64_t offset, uint64_t seed,
                          uint64_t tensor_id, double mean, double sigma, int fp16) {
  uint64_t key = ssdi_key(seed, tensor_id);
  int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < nn; ++k) out[k] = value_bits(key, offset + (uint64_t)k, mean, sigma, fp16);
}

/* out[i] = bits of the 16-bit constant c (e.g. a unit RMSNorm gain). */
void ssd_inputs_fill_const_host(uint16_t* out, uint64_t n, float c, int fp16) {
  uint16_t b;
  if (fp16) {
    union { _Float16 h; uint16_t u; } v;
    v.h = (_Float16)c;
    b = v.u;
  } else {
    b = ssdi_f32_to_bf16_bits(c);
  }
  for (uint64_t k = 0; k < n; ++k) out[k] = b;
}

/* Uniform random prompt token ids in [0, vocab). */
void ssd_inputs_prompt_host(int32_t* out, int n, uint64_t seed, int vocab) {
  uint64_t key = ssdi_key(seed, SSDI_PROMPT_ID);
  for (int i = 0; i < n; ++i) out[i] = (int32_t)(ssdi_mix(key + (uint64_t)i) % (uint64_t)vocab);
}

/* The raw counter hash, exported so tests can check it against SplitMix64's published outputs. */
uint64_t ssd_inputs_mix_host(uint64_t x) { return ssdi_mix(x); }
