// ssd_attention_noalloc: the attention entry point for callers that cannot
// allocate device memory.  Its scratch (the row descriptor; the split merge
// runs in distributed shared memory and needs none) lives in a file-scope
// __device__ array that every GPU loading this library holds until the
// process exits; the call itself is ssd_attention on that array.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/ssd.h"
#include "common.cuh"

namespace {

constexpr size_t kNoAllocBytes = 4096;  // per device: one row descriptor (rounded up to 256 bytes)
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_attn_scratch[kNoAllocBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_attn_scratch on the current device, looked up once per
// device with that device current.  In host code the array's name is only a
// stand-in for the symbol, never a usable device address.
ssd_status scratch_for_device(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return SSD_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) return SSD_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SSD_OK;
}

}  // namespace

extern "C" ssd_status ssd_attention_noalloc(const ssd_attention_args* a, void* stream) {
  static_assert(sizeof(ssd::PassDesc) <= kNoAllocBytes, "the row descriptor must fit the static array");
  if (!a) return SSD_ERR_INVALID_ARG;
  int cur = 0, sdev = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) return SSD_ERR_CUDA;
  // the array's address belongs to the current device: the stream must be on that device too
  if (cudaStreamGetDevice((cudaStream_t)stream, &sdev) != cudaSuccess) {
    cudaGetLastError();
    return SSD_ERR_INVALID_ARG;
  }
  if (sdev != cur) return SSD_ERR_INVALID_ARG;
  void* base = nullptr;
  const ssd_status s = scratch_for_device(cur, &base);
  if (s != SSD_OK) return s;
  return ssd_attention(a, base, kNoAllocBytes, stream);
}
