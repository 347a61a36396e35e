/*
 * Device fill kernel for the seeded synthetic inputs (definition in
 * gen_def.h).  It writes the same 16-bit values as gen_host.c straight into
 * device memory, so multi-GB weight sets never cross PCIe/C2C.  Built as
 * libssd_inputs_dev.so; no part of the decoding method.
 */
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gen_def.h"

__global__ void ssdi_fill_kernel(uint16_t* __restrict__ out, uint64_t n, uint64_t offset, uint64_t key,
                                 double mean, double sigma, int fp16) {
  const double two_pi = 6.283185307179586476925286766559;
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t k = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n; k += stride) {
    uint64_t i = offset + k;
    uint64_t r1 = ssdi_mix(key + 2 * i);
    uint64_t r2 = ssdi_mix(key + 2 * i + 1);
    double z = sqrt(-2.0 * log(ssdi_u1(r1))) * cos(two_pi * ssdi_u2(r2));
    float f = (float)(mean + sigma * z);
    if (fp16) {
      __half h = __float2half_rn(f);
      out[k] = *reinterpret_cast<uint16_t*>(&h);
    } else {
      out[k] = ssdi_f32_to_bf16_bits(f);
    }
  }
}

__global__ void ssdi_const_kernel(uint16_t* __restrict__ out, uint64_t n, uint16_t bits) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t k = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n; k += stride) out[k] = bits;
}

static int grid_for(uint64_t n) {
  uint64_t g = (n + 255) / 256;
  if (g > 152ull * 16) g = 152ull * 16;
  if (g < 1) g = 1;
  return (int)g;
}

extern "C" int ssd_inputs_fill_dev(void* dptr, uint64_t n, uint64_t offset, uint64_t seed, uint64_t tensor_id,
                                   double mean, double sigma, int fp16, void* stream) {
  if (n == 0) return 0;
  if (dptr == nullptr) return 1;
  ssdi_fill_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>((uint16_t*)dptr, n, offset,
                                                                   ssdi_key(seed, tensor_id), mean, sigma, fp16);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

extern "C" int ssd_inputs_fill_const_dev(void* dptr, uint64_t n, float c, int fp16, void* stream) {
  if (n == 0) return 0;
  if (dptr == nullptr) return 1;
  uint16_t bits;
  if (fp16) {
    __half h = __float2half_rn(c);
    bits = *reinterpret_cast<uint16_t*>(&h);
  } else {
    bits = ssdi_f32_to_bf16_bits(c);
  }
  ssdi_const_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>((uint16_t*)dptr, n, bits);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
