// Shared device-side definitions of libssd: pass descriptor, device state,
// 16-bit load/convert helpers, warp reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssd {

constexpr int kMaxRows = 64;     // rows one pass may carry (uint64 visibility masks)
constexpr int kPage = 64;        // KV-cache page size in tokens
constexpr int kMaxLayers = 128;

// Per-pass row description, built on the device at the start of each pass
// from the committed length, so captured graphs replay at any position.
// Row r runs at RoPE position pos[r], writes its K/V to cache slot slot[r],
// and sees cache slots [0, prefix) plus slots base + e for every bit e set in
// mask[r] (the "special mask" that lets draft/verify/tree/DP rows share one
// KV cache without duplicating it).
struct PassDesc {
  int rows;
  int prefix;
  int base;
  int pad_;
  int pos[kMaxRows];
  int slot[kMaxRows];
  unsigned long long mask[kMaxRows];
};

// Request state that lives on the device so whole decode cycles run without
// host round trips.
constexpr int kDevErrToken = 3;  // DevState::err: a token id past the vocabulary reached the embedding

struct DevState {
  int t;          // committed length
  int pending;    // pending token (emitted, not yet in the cache)
  int gen_count;  // tokens written to out_tokens by the current generate call
  int gen_cap;    // capacity of out_tokens
  int n_acc;      // accepted drafts in the last verify
  int bonus;      // bonus token of the last verify
  int tgt_row;    // stash row holding the CLaSp target (last accepted token)
  int tgt_pos;    // its position
  int exp_idx;    // DyTC: index of the next tree expansion
  int err;        // device-side error flag: 0 ok, 1-2 a bounded wait gave up, kDevErrToken a bad token id
  int last_path_len;
  // Draft exit (linear drafts with a confidence threshold): draft_live is 1 while
  // drafting goes on and 0 once a draft's top-1 probability fell below the
  // threshold; draft_n = drafts written by the current draft pass.
  int draft_live;
  int draft_n;
  int path[kMaxRows + 1];
  long long cycles, accepted;
  long long hist[kMaxRows + 1];
  long long drafted;            // draft rows verified (padding rows after a draft exit not counted)
  float draft_p1[kMaxRows];     // top-1 softmax probability of each draft of the last exit-enabled draft pass
};

template <typename T>
struct Io;

template <>
struct Io<__nv_bfloat16> {
  static __device__ __forceinline__ void unpack8(const uint4& u, float f[8]) {
    f[0] = __uint_as_float(u.x << 16);
    f[1] = __uint_as_float(u.x & 0xffff0000u);
    f[2] = __uint_as_float(u.y << 16);
    f[3] = __uint_as_float(u.y & 0xffff0000u);
    f[4] = __uint_as_float(u.z << 16);
    f[5] = __uint_as_float(u.z & 0xffff0000u);
    f[6] = __uint_as_float(u.w << 16);
    f[7] = __uint_as_float(u.w & 0xffff0000u);
  }
  static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

template <>
struct Io<__half> {
  static __device__ __forceinline__ void unpack8(const uint4& u, float f[8]) {
    const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 v = __half22float2(h[i]);
      f[2 * i] = v.x;
      f[2 * i + 1] = v.y;
    }
  }
  static __device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
  static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
};

// 16-byte streaming load that bypasses L1 allocation (weights are read once).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Per-token int8 code of x given m = 127 / amax (IEEE float32 division done
// by the caller): round-half-even of the float32 product, clamped to +-127.
__device__ __forceinline__ float q8_code(float x, float m) {
  float c = rintf(__fmul_rn(x, m));
  return fminf(127.f, fmaxf(-127.f, c));
}

// KV-cache address of (layer, slot, kv head, dim): pages of kPage tokens,
// layout [layer][page][kv head][kPage][head_dim].
__device__ __forceinline__ size_t kv_index(int layer, int slot, int kvh, int d, const int* btab, int n_pages,
                                           int n_kv, int hd) {
  int page = btab[slot / kPage];
  return ((((size_t)layer * n_pages + page) * n_kv + kvh) * kPage + (slot % kPage)) * hd + d;
}

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(phase)
      : "memory");
  return ok != 0;
}

// Wait for an mbarrier phase with an iteration limit (each try_wait may block
// for a short hardware-defined time); false if the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t phase) {
  for (uint32_t i = 0; i < (1u << 22); ++i)
    if (mbar_try_wait(bar, phase)) return true;
  return false;
}

// Bulk (non-tensor) TMA copy global -> this CTA's shared memory, completing on `bar`.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before later async-proxy writes.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Prefetch this CTA's share (part of nparts) of [p, p + bytes) into L2 with
// bulk prefetches of at most 64 KB, one per thread.  p 16-byte aligned.
__device__ __forceinline__ void l2_prefetch_share(const void* p, size_t bytes, int part, int nparts) {
  if (!p || bytes == 0) return;
  const size_t per = ((bytes + nparts - 1) / nparts + 15) & ~(size_t)15;
  const size_t b0 = per * part;
  if (b0 >= bytes) return;
  const size_t b1 = b0 + per < bytes ? b0 + per : bytes;
  for (size_t o = b0 + (size_t)threadIdx.x * 65536; o < b1; o += (size_t)blockDim.x * 65536) {
    const size_t n = (b1 - o < 65536 ? b1 - o : 65536) & ~(size_t)15;
    if (n)
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"((const char*)p + o), "r"((uint32_t)n)
                   : "memory");
  }
}

// Draft exit gate: a kernel of a later draft forward receives &DevState::draft_live
// (null: no gate).  Read before griddep_wait() it is only a hint (whether to
// warm caches early); read after it, it decides whether the kernel runs: the
// word is written only by kernels that completed before the wait returned, so
// every CTA of the launch reads the same value.
__device__ __forceinline__ bool gate_open(const int* g) {
  return g == nullptr || *reinterpret_cast<const volatile int*>(g) != 0;
}

// Kernel timeline tracing (SSD_OPT_TRACE): slot = {~min(resident), ~min(running), max(end)}
// of %globaltimer over the launch's CTAs; a zeroed slot is the neutral value.
__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void trace_mark(unsigned long long* tr, int which) {
  if (tr && threadIdx.x == 0) {
    const unsigned long long t = gtimer();
    atomicMax(tr + which, which == 2 ? t : ~t);
  }
}

// Programmatic dependent launch: wait until the preceding kernel in the stream
// has completed and its writes are visible (a no-op when launched normally) /
// allow the next kernel to start launching.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace ssd
