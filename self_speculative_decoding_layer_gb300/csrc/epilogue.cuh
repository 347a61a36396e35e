// Epilogues shared by the projection kernels (CUDA-core and tensor-core):
// what happens to the result y of a pair of weight rows for one input row.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace ssd {

template <typename T>
__device__ __forceinline__ void epi_apply(const LinearArgs& a, int m, int u, float y0, float y1) {
  const int mg = a.row0 + m;  // row within the pass
  if (a.epi == EPI_QKV) {
    const int half = a.hd >> 1;
    const int head = u / half, i = u - head * half;
    const int pos = a.desc->pos[mg];
    if (head < a.n_q + a.n_kv) {  // RoPE (rotate-half) on q and k
      const float c = a.rope_cos[(size_t)pos * half + i], s = a.rope_sin[(size_t)pos * half + i];
      const float z0 = y0 * c - y1 * s, z1 = y1 * c + y0 * s;
      y0 = z0;
      y1 = z1;
    }
    if (head < a.n_q) {
      float* q = a.out + (size_t)m * a.ldo + head * a.hd;
      q[i] = y0;
      q[i + half] = y1;
    } else {
      const bool is_k = head < a.n_q + a.n_kv;
      const int kvh = is_k ? head - a.n_q : head - a.n_q - a.n_kv;
      const int slot = a.desc->slot[mg];
      float* c = reinterpret_cast<float*>(is_k ? a.kcache : a.vcache);  // the KV cache is fp32
      size_t base = kv_index(a.layer, slot, kvh, 0, a.btab, a.n_pages, a.n_kv, a.hd);
      c[base + i] = y0;
      c[base + i + half] = y1;
    }
  } else if (a.epi == EPI_RESID) {
    float* h = a.out + (size_t)m * a.ldo + 2 * u;
    const float h0 = h[0] + y0, h1 = h[1] + y1;
    h[0] = h0;
    h[1] = h1;
    if (a.stash) {
      float* s = a.stash + (size_t)m * a.ldo + 2 * u;
      s[0] = h0;
      s[1] = h1;
    }
  } else if (a.epi == EPI_SWIGLU) {
    const float g = y0 / (1.0f + expf(-y0));
    const float v = g * y1;
    a.out[(size_t)m * a.ldo + u] = v;
    if (a.xb_next) {  // the down projection's operand rows: v = hi + lo
      T* xb = reinterpret_cast<T*>(a.xb_next);
      const T hi = Io<T>::from_f(v);
      xb[(size_t)m * a.F + u] = hi;
      xb[((size_t)a.next_mp + m) * a.F + u] = Io<T>::from_f(v - Io<T>::to_f(hi));
    }
  } else {
    float* o = a.out + (size_t)m * a.ldo + 2 * u;
    o[0] = y0;
    o[1] = y1;
  }
}

__device__ __forceinline__ int n_units(const LinearArgs& a) { return a.epi == EPI_SWIGLU ? a.F : a.N / 2; }

__device__ __forceinline__ void unit_rows(const LinearArgs& a, int u, int& r0, int& r1) {
  if (a.epi == EPI_QKV) {
    const int half = a.hd >> 1, head = u / half;
    r0 = head * a.hd + (u - head * half);
    r1 = r0 + half;
  } else if (a.epi == EPI_SWIGLU) {
    r0 = u;
    r1 = a.F + u;
  } else {
    r0 = 2 * u;
    r1 = 2 * u + 1;
  }
}

}  // namespace ssd
