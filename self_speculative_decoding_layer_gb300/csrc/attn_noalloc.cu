// ssd_attention_noalloc: the attention entry point for callers that cannot
// allocate device memory.  Its scratch (the row descriptor; the split merge
// runs in distributed shared memory and needs none) lives in a file-scope
// __device__ array that every GPU loading this library holds until the
// process exits.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "../../include/ssd.h"
#include "common.cuh"
#include "kernels.h"

using namespace ssd;

namespace {

constexpr size_t kNoAllocBytes = 4096;  // per device: one row descriptor
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_attn_scratch[kNoAllocBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_attn_scratch on the current device, looked up once per
// device.  In host code the array's name is only a stand-in for the symbol,
// never a usable device address.
ssd_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSD_ERR_CUDA;
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
  if (!a || !a->q || !a->k_cache || !a->v_cache || !a->block_table || !a->out) return SSD_ERR_INVALID_ARG;
  if (a->rows < 1 || a->rows > kMaxRows || a->n_q_heads < 1 || a->n_kv_heads < 1 ||
      a->n_q_heads % a->n_kv_heads || (a->head_dim != 64 && a->head_dim != 128))
    return SSD_ERR_INVALID_ARG;
  if (a->prefix < 0 || a->base < 0 || a->layer < 0 || a->n_pages < 1) return SSD_ERR_INVALID_ARG;
  if (a->dtype < SSD_BF16 || a->dtype > SSD_F32) return SSD_ERR_INVALID_ARG;
  if (((uintptr_t)a->k_cache | (uintptr_t)a->v_cache | (uintptr_t)a->q | (uintptr_t)a->out) & 15)
    return SSD_ERR_INVALID_ARG;  // 16-byte vector and TMA accesses
  if ((int64_t)a->prefix > (int64_t)a->n_pages * kPage || (int64_t)a->base + a->rows > (int64_t)a->n_pages * kPage)
    return SSD_ERR_INVALID_ARG;
  static_assert(sizeof(PassDesc) <= kNoAllocBytes, "the row descriptor must fit the static array");
  void* base = nullptr;
  ssd_status s = scratch_for_current_device(&base);
  if (s != SSD_OK) return s;

  PassDesc d{};
  d.rows = a->rows;
  d.prefix = a->prefix;
  d.base = a->base;
  for (int r = 0; r < a->rows; ++r) d.mask[r] = a->mask[r];
  PassDesc* dd = (PassDesc*)base;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(dd, &d, sizeof(d), cudaMemcpyHostToDevice, st) != cudaSuccess) return SSD_ERR_CUDA;
  AttnArgs b{};
  b.desc = dd;
  b.q = a->q;
  b.kcache = a->k_cache;
  b.vcache = a->v_cache;
  b.btab = a->block_table;
  b.n_pages = a->n_pages;
  b.layer = a->layer;
  b.n_q = a->n_q_heads;
  b.n_kv = a->n_kv_heads;
  b.hd = a->head_dim;
  b.out = a->out;
  b.rows = a->rows;
  attention_layout(a->prefix + a->rows, a->rows, a->n_q_heads / a->n_kv_heads, a->n_kv_heads, a->dtype, a->head_dim,
                   &b.qb, &b.n_split);
  b.max_keys = a->prefix + a->rows;
  g_pdl = false;
  if (!launch_attention(b, a->dtype, st)) return SSD_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}
