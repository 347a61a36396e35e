/*
 * Seeded synthetic inputs: one definition, used by the host generator
 * (gen_host.c, for the CPU oracle) and by the device fill kernel
 * (gen_dev.cu, for the GPU path).  This header holds no arithmetic of the
 * decoding method itself: only a counter-based random stream and the
 * Box-Muller transform that turn (seed, tensor id, element index) into a
 * weight value or a prompt token.
 *
 * Definitions (all arithmetic is exact integer or IEEE double/float; both
 * implementations are compiled without multiply-add contraction):
 *   mix(x)        = SplitMix64 output function applied to x + golden gamma
 *                   (Steele, Lea, Flood, "Fast splittable pseudorandom number
 *                   generators", OOPSLA 2014).
 *   key(seed,id)  = mix(seed ^ mix(id))
 *   r1, r2        = mix(key + 2*i), mix(key + 2*i + 1)      for element i
 *   u1            = ((r1 >> 11) + 1) * 2^-53                 in (0, 1]
 *   u2            =  (r2 >> 11)      * 2^-53                 in [0, 1)
 *   z             = sqrt(-2 ln u1) * cos(2 pi u2)            (Box-Muller 1958)
 *   value         = round_to_16bit( (float)(mean + sigma * z) ) float RNE, then
 *                   bf16 RNE (bit trick below) or fp16 RNE (IEEE conversion)
 *   prompt tok i  = mix(key(seed, PROMPT_ID) + i) mod vocab
 */
#ifndef SSD_INPUTS_GEN_DEF_H
#define SSD_INPUTS_GEN_DEF_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SSDI_FN static __host__ __device__ __forceinline__
#else
#define SSDI_FN static inline
#endif

#define SSDI_PROMPT_ID 0x50524F4D50540000ULL /* "PROMPT" */

SSDI_FN uint64_t ssdi_mix(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

SSDI_FN uint64_t ssdi_key(uint64_t seed, uint64_t id) { return ssdi_mix(seed ^ ssdi_mix(id)); }

SSDI_FN double ssdi_u1(uint64_t r) { return (double)((r >> 11) + 1) * (1.0 / 9007199254740992.0); }
SSDI_FN double ssdi_u2(uint64_t r) { return (double)(r >> 11) * (1.0 / 9007199254740992.0); }

/* float -> bf16 bits, round to nearest even (inputs here are finite) */
SSDI_FN uint16_t ssdi_f32_to_bf16_bits(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  uint32_t u = v.u;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

#endif
