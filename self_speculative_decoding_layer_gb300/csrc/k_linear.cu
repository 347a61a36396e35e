// CUDA-core linear kernels: y = W x for small row counts, with the fused
// RMSNorm / int8 prologue and the QKV-RoPE-KV / residual / SwiGLU / logits
// epilogues shared by every projection of the decoder layer.
//
// k_gemv_rs is the batch-1 (one row) weight-streaming kernel used by
// autoregressive steps and linear drafts.  Built with SSD_CROSSCHECK (the
// test library only) the file also holds the cross-check kernels: the
// general CUDA-core rows kernel k_linear_rows (any row count, the
// tensor-core path's reference) and two other batch-1 GEMVs (k_gemv one
// row pair per warp, k_gemv_bulk TMA-bulk stream-K).
#include <math.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace ssd {

// Per-row prologue statistics: s_inv[m] = 1/sqrt(mean(x^2)+eps) (1 without
// a norm), s_qm[m] = 127/amax and s_qs[m] = amax/127 of the normalised row
// (int8 only).  All threads of the block cooperate on each row (16-byte
// loads, block-wide reductions), so the weight stream is not held up by a
// long serial walk over the input row.  The caller synchronises afterwards.
__device__ __forceinline__ float block_reduce(float v, float* red, bool is_max) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  v = is_max ? warp_max(v) : warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
  for (int w = 1; w < nw; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
  return r;
}

template <typename T>
__device__ void row_stats(const LinearArgs& a, int m0, int nrows, float* s_inv, float* s_qm, float* s_qs) {
  __shared__ float red[32];
  const T* g = reinterpret_cast<const T*>(a.gamma);
  for (int m = 0; m < nrows; ++m) {
    const float* x = a.X + (size_t)(m0 + m) * a.ldx;
    float inv = 1.0f;
    if (g) {
      float ss = 0.f;
      for (int k = threadIdx.x * 8; k < a.K; k += blockDim.x * 8) {
        const float4* xp = reinterpret_cast<const float4*>(x + k);
        const float4 u = xp[0], v = xp[1];
        ss += u.x * u.x + u.y * u.y + u.z * u.z + u.w * u.w + v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
      }
      ss = block_reduce(ss, red, false);
      inv = 1.0f / sqrtf(ss / (float)a.K + a.eps);
    }
    float qm = 0.f, qs = 0.f;
    if (a.int8) {
      float amax = 0.f;
      for (int k = threadIdx.x * 8; k < a.K; k += blockDim.x * 8) {
        const float4* xp = reinterpret_cast<const float4*>(x + k);
        const float4 u = xp[0], v = xp[1];
        float xv[8] = {u.x, u.y, u.z, u.w, v.x, v.y, v.z, v.w};
        float gv[8];
        if (g) Io<T>::unpack8(*reinterpret_cast<const uint4*>(g + k), gv);
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(g ? xv[e] * inv * gv[e] : xv[e]));
      }
      amax = block_reduce(amax, red, true);
      if (amax > 0.f) {
        qm = __fdiv_rn(127.0f, amax);
        qs = __fdiv_rn(amax, 127.0f);
      }
    }
    if (threadIdx.x == 0) {
      s_inv[m] = inv;
      s_qm[m] = qm;
      s_qs[m] = qs;
    }
  }
}

// Normalise / quantize 8 consecutive inputs of row m in place.
template <typename T>
__device__ __forceinline__ void prep8(const LinearArgs& a, float x[8], const float g[8], float inv, float qm) {
  if (a.gamma) {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = x[j] * inv * g[j];
  }
  if (a.int8) {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = q8_code(x[j], qm);
  }
}

#ifdef SSD_CROSSCHECK
// Cross-check kernels (built into the test library only): the general CUDA-core rows kernel and
// the per-row-pair batch-1 GEMV, against which the tensor-core and stream-K paths are compared.
// ---------------------------------------------------------------- rows kernel

template <typename T, int MT>
__global__ void __launch_bounds__(256) k_linear_rows(LinearArgs a) {
  __shared__ float s_inv[MT], s_qm[MT], s_qs[MT];
  griddep_launch();
  trace_mark(a.trace, 0);
  griddep_wait();
  if (!gate_open(a.gate)) return;
  trace_mark(a.trace, 1);
  row_stats<T>(a, 0, a.M, s_inv, s_qm, s_qs);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const T* W = reinterpret_cast<const T*>(a.W);
  const T* G = reinterpret_cast<const T*>(a.gamma);
  const int nu = n_units(a);
  for (int u = blockIdx.x * 8 + warp; u < nu; u += gridDim.x * 8) {
    int r0, r1;
    unit_rows(a, u, r0, r1);
    float acc0[MT], acc1[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc0[m] = acc1[m] = 0.f;
    const T* w0p = W + (size_t)r0 * a.K;
    const T* w1p = W + (size_t)r1 * a.K;
    for (int k = lane * 8; k < a.K; k += 256) {
      float w0[8], w1[8], g[8];
      Io<T>::unpack8(ld_stream16(w0p + k), w0);
      Io<T>::unpack8(ld_stream16(w1p + k), w1);
      if (G) Io<T>::unpack8(__ldg(reinterpret_cast<const uint4*>(G + k)), g);
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m < a.M) {
          const float4* xp = reinterpret_cast<const float4*>(a.X + (size_t)m * a.ldx + k);
          float4 xa = __ldg(xp), xb = __ldg(xp + 1);
          float x[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
          prep8<T>(a, x, g, s_inv[m], s_qm[m]);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            acc0[m] = fmaf(w0[j], x[j], acc0[m]);
            acc1[m] = fmaf(w1[j], x[j], acc1[m]);
          }
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m < a.M) {
        float y0 = warp_sum(acc0[m]), y1 = warp_sum(acc1[m]);
        if (lane == (m & 31)) {
          if (a.int8) {
            y0 *= s_qs[m];
            y1 *= s_qs[m];
          }
          epi_apply<T>(a, m, u, y0, y1);
        }
      }
    }
  }
  __syncthreads();
  trace_mark(a.trace, 2);
}

template <typename T, int MT>
static void run_rows(const LinearArgs& a, cudaStream_t st) {
  int units = a.epi == EPI_SWIGLU ? a.F : a.N / 2;
  int grid = (units + 7) / 8;
  if (grid > 152 * 8) grid = 152 * 8;
  launch_ex(k_linear_rows<T, MT>, dim3(grid), dim3(256), 0, st, a);
}

template <typename T>
static void rows_dispatch(const LinearArgs& a0, cudaStream_t st) {
  for (int m0 = 0; m0 < a0.M; m0 += 32) {
    LinearArgs a = a0;
    a.M = a0.M - m0 < 32 ? a0.M - m0 : 32;
    a.X = a0.X + (size_t)m0 * a0.ldx;
    a.row0 = a0.row0 + m0;
    a.out = a0.out + (size_t)m0 * a0.ldo;
    if (a0.stash) a.stash = a0.stash + (size_t)m0 * a0.ldo;
    if (a.M == 1)
      run_rows<T, 1>(a, st);
    else if (a.M <= 2)
      run_rows<T, 2>(a, st);
    else if (a.M <= 4)
      run_rows<T, 4>(a, st);
    else if (a.M <= 8)
      run_rows<T, 8>(a, st);
    else if (a.M <= 16)
      run_rows<T, 16>(a, st);
    else
      run_rows<T, 32>(a, st);
  }
}

void launch_linear_rows(const LinearArgs& a, int fp16, cudaStream_t st) {
  if (fp16)
    rows_dispatch<__half>(a, st);
  else
    rows_dispatch<__nv_bfloat16>(a, st);
}

// ---------------------------------------------------------------- batch-1 GEMV
//
// One input row.  The prologue normalises / quantizes x once per CTA into
// shared memory (at most ffn floats), then each warp streams two weight rows
// per unit with 16-byte loads, four loads in flight per row.

template <typename T>
__global__ void __launch_bounds__(256) k_gemv(LinearArgs a) {
  extern __shared__ float s_x[];
  __shared__ float s_inv[1], s_qm[1], s_qs[1];
  griddep_launch();
  trace_mark(a.trace, 0);
  griddep_wait();
  if (!gate_open(a.gate)) return;
  trace_mark(a.trace, 1);
  row_stats<T>(a, 0, 1, s_inv, s_qm, s_qs);
  __syncthreads();
  const T* G = reinterpret_cast<const T*>(a.gamma);
  const float inv = s_inv[0], qm = s_qm[0];
  for (int k = threadIdx.x * 8; k < a.K; k += blockDim.x * 8) {
    const float4* xp = reinterpret_cast<const float4*>(a.X + k);
    float4 xa = xp[0], xb = xp[1];
    float x[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
    float g[8];
    if (G) Io<T>::unpack8(*reinterpret_cast<const uint4*>(G + k), g);
    prep8<T>(a, x, g, inv, qm);
    float4* sp = reinterpret_cast<float4*>(s_x + k);
    sp[0] = make_float4(x[0], x[1], x[2], x[3]);
    sp[1] = make_float4(x[4], x[5], x[6], x[7]);
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const T* W = reinterpret_cast<const T*>(a.W);
  const int nu = n_units(a);
  const int K = a.K;
  for (int u = blockIdx.x * 8 + warp; u < nu; u += gridDim.x * 8) {
    int r0, r1;
    unit_rows(a, u, r0, r1);
    const T* w0p = W + (size_t)r0 * K;
    const T* w1p = W + (size_t)r1 * K;
    float acc0 = 0.f, acc1 = 0.f;
    int k = lane * 8;
    for (; k + 3 * 256 < K; k += 4 * 256) {
      uint4 u0[4], u1[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        u0[j] = ld_stream16(w0p + k + j * 256);
        u1[j] = ld_stream16(w1p + k + j * 256);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float w0[8], w1[8];
        Io<T>::unpack8(u0[j], w0);
        Io<T>::unpack8(u1[j], w1);
        const float4* sp = reinterpret_cast<const float4*>(s_x + k + j * 256);
        float4 xa = sp[0], xb = sp[1];
        float x[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          acc0 = fmaf(w0[e], x[e], acc0);
          acc1 = fmaf(w1[e], x[e], acc1);
        }
      }
    }
    for (; k < K; k += 256) {
      float w0[8], w1[8];
      Io<T>::unpack8(ld_stream16(w0p + k), w0);
      Io<T>::unpack8(ld_stream16(w1p + k), w1);
      const float4* sp = reinterpret_cast<const float4*>(s_x + k);
      float4 xa = sp[0], xb = sp[1];
      float x[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        acc0 = fmaf(w0[e], x[e], acc0);
        acc1 = fmaf(w1[e], x[e], acc1);
      }
    }
    float y0 = warp_sum(acc0), y1 = warp_sum(acc1);
    if (lane == 0) {
      if (a.int8) {
        y0 *= s_qs[0];
        y1 *= s_qs[0];
      }
      epi_apply<T>(a, 0, u, y0, y1);
    }
  }
  __syncthreads();
  trace_mark(a.trace, 2);
}

template <typename T>
static void run_gemv(const LinearArgs& a, cudaStream_t st) {
  int units = a.epi == EPI_SWIGLU ? a.F : a.N / 2;
  int grid = (units + 7) / 8;
  const int per_sm = a.K * 4 <= 48 * 1024 ? 4 : (a.K * 4 <= 72 * 1024 ? 3 : 1);
  if (grid > 152 * per_sm) grid = 152 * per_sm;
  launch_ex(k_gemv<T>, dim3(grid), dim3(256), (size_t)a.K * sizeof(float), st, a);
}
#endif  // SSD_CROSSCHECK

// ---------------------------------------------------------------- batch-1 GEMV, TMA-bulk stream-K
//
// Each warp owns an equal, contiguous slice of the (row pair, 1024-element
// chunk) steps of the whole matrix, so every warp moves the same number of
// bytes whatever the row count.  Lane 0 of the warp keeps NS chunk pairs in
// flight with cp.async.bulk into a per-warp shared-memory ring (one mbarrier
// per stage); the 32 lanes consume each stage against x held in shared
// memory.  A row pair cut by a slice boundary belongs to two warps (every
// slice here is at least one row pair long); gemv_finish merges it.  The first NS
// stages are requested before griddepcontrol.wait, so under programmatic
// dependent launch the weight stream starts while the previous kernel drains.

constexpr int kCK = 1024;
constexpr int kGW = 8;  // warps per CTA

// Finish a warp's segment [c0, c1) of unit u (the unit's K range in chunks
// of kCK; nchunks per unit) with the partial dot products y0, y1 of the
// unit's two rows.  nw warps split the (unit, chunk) slices evenly,
// so a unit may span several warps: each writes its partials to the unit's
// slot c0, and the warp whose chunks complete the unit sums the segments in
// slice order (deterministic whichever warp comes last) and runs the epilogue.
template <typename T>
__device__ __forceinline__ void gemv_finish(const LinearArgs& a, int u, int c0, int c1, int nchunks, int nw, float y0,
                                            float y1, float qs) {
  if (c1 - c0 < nchunks) {
    const long long total = (long long)n_units(a) * nchunks;
    float* p = a.sk_part + ((size_t)u * nchunks + c0) * 2;
    p[0] = y0;
    p[1] = y1;
    __threadfence();
    const int prev = atomicAdd(a.sk_cnt + u, c1 - c0);
    if (prev + (c1 - c0) < nchunks) return;
    __threadfence();
    const long long sa = (long long)u * nchunks;
    const int g0 = (int)(((sa + 1) * nw - 1) / total);        // warp holding the unit's first slice
    const int g1 = (int)(((sa + nchunks) * nw - 1) / total);  // ... and its last
    y0 = 0.f;
    y1 = 0.f;
    for (int g = g0; g <= g1; ++g) {
      const long long sg = total * g / nw;
      const float* q = a.sk_part + ((size_t)u * nchunks + (sg > sa ? (int)(sg - sa) : 0)) * 2;
      y0 += __ldcg(q);
      y1 += __ldcg(q + 1);
    }
    a.sk_cnt[u] = 0;
  }
  if (a.int8) {
    y0 *= qs;
    y1 *= qs;
  }
  epi_apply<T>(a, 0, u, y0, y1);
}

#ifdef SSD_CROSSCHECK
template <typename T, int NS>
__global__ void __launch_bounds__(256, 1) k_gemv_bulk(LinearArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float s_inv[1], s_qm[1], s_qs[1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = a.K;
  const size_t xbytes = ((size_t)K * 4 + 127) & ~(size_t)127;
  float* s_x = reinterpret_cast<float*>(smem);
  T* ring = reinterpret_cast<T*>(smem + xbytes) + (size_t)warp * NS * 2 * kCK;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + xbytes + (size_t)kGW * NS * 2 * kCK * sizeof(T)) + warp * NS;

  griddep_launch();
  const int nu = n_units(a);
  const int nchunks = (K + kCK - 1) / kCK;
  const long long total = (long long)nu * nchunks;
  const int nw = min((int)gridDim.x * kGW, nu);
  const int gw = blockIdx.x * kGW + warp;
  long long s0 = 0, s1 = 0;
  if (gw < nw) {
    s0 = total * gw / nw;
    s1 = total * (gw + 1) / nw;
  }
  const int len = (int)(s1 - s0);
  const T* W = reinterpret_cast<const T*>(a.W);

  if (lane == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
  }
  __syncwarp();

  auto issue = [&](int ls) {
    const long long s = s0 + ls;
    const int u = (int)(s / nchunks), c = (int)(s - (long long)u * nchunks);
    int r0, r1;
    unit_rows(a, u, r0, r1);
    const int k0 = c * kCK;
    const int n = min(kCK, K - k0);
    const uint32_t bytes = (uint32_t)n * (uint32_t)sizeof(T);
    T* dst = ring + (size_t)(ls % NS) * 2 * kCK;
    uint64_t* bar = &bars[ls % NS];
    mbar_expect_tx(bar, 2 * bytes);
    bulk_g2s(dst, W + (size_t)r0 * K + k0, bytes, bar);
    bulk_g2s(dst + kCK, W + (size_t)r1 * K + k0, bytes, bar);
  };
  // the first NS steps' copies go out before the wait, unless a draft exit has already closed the gate
  const bool warm = gate_open(a.gate);
  if (lane == 0 && warm)
    for (int ls = 0; ls < min(NS, len); ++ls) issue(ls);

  trace_mark(a.trace, 0);
  griddep_wait();
  if (!gate_open(a.gate)) {  // nothing to do: let the copies already issued land before the CTA exits
    if (lane == 0 && warm)
      for (int ls = 0; ls < min(NS, len); ++ls) mbar_wait_bounded(&bars[ls], 0u);
    return;
  }
  if (lane == 0 && !warm)
    for (int ls = 0; ls < min(NS, len); ++ls) issue(ls);
  trace_mark(a.trace, 1);
  row_stats<T>(a, 0, 1, s_inv, s_qm, s_qs);
  __syncthreads();
  {
    const T* G = reinterpret_cast<const T*>(a.gamma);
    const float inv = s_inv[0], qm = s_qm[0];
    for (int k = threadIdx.x * 8; k < K; k += blockDim.x * 8) {
      const float4* xp = reinterpret_cast<const float4*>(a.X + k);
      float4 xa = xp[0], xb = xp[1];
      float x[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
      float g[8];
      if (G) Io<T>::unpack8(*reinterpret_cast<const uint4*>(G + k), g);
      prep8<T>(a, x, g, inv, qm);
      float4* sp = reinterpret_cast<float4*>(s_x + k);
      sp[0] = make_float4(x[0], x[1], x[2], x[3]);
      sp[1] = make_float4(x[4], x[5], x[6], x[7]);
    }
  }
  __syncthreads();
  const float qs = s_qs[0];

  float acc0 = 0.f, acc1 = 0.f;
  int ls = 0;
  bool ok = true;
  for (; ls < len; ++ls) {
    const long long s = s0 + ls;
    const int u = (int)(s / nchunks), c = (int)(s - (long long)u * nchunks);
    const int k0 = c * kCK, n = min(kCK, K - k0);
    if (!mbar_wait_bounded(&bars[ls % NS], (uint32_t)((ls / NS) & 1))) {
      ok = false;
      break;
    }
    const T* w0 = ring + (size_t)(ls % NS) * 2 * kCK;
    const T* w1 = w0 + kCK;
    const float* xs = s_x + k0;
#pragma unroll 2
    for (int e = lane * 8; e < n; e += 256) {
      float f0[8], f1[8];
      Io<T>::unpack8(*reinterpret_cast<const uint4*>(w0 + e), f0);
      Io<T>::unpack8(*reinterpret_cast<const uint4*>(w1 + e), f1);
      const float4* xp = reinterpret_cast<const float4*>(xs + e);
      const float4 xa = xp[0], xb = xp[1];
      const float x[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        acc0 = fmaf(f0[j], x[j], acc0);
        acc1 = fmaf(f1[j], x[j], acc1);
      }
    }
    __syncwarp();
    if (lane == 0 && ls + NS < len) {
      fence_proxy_async();
      issue(ls + NS);
    }
    if (c == nchunks - 1 || ls == len - 1) {
      const float y0 = warp_sum(acc0), y1 = warp_sum(acc1);
      acc0 = acc1 = 0.f;
      if (lane == 0)
        gemv_finish<T>(a, u, (s - c) >= s0 ? 0 : (int)(s0 - (s - c)), c + 1, nchunks, nw, y0, y1, qs);
    }
  }
  if (!ok) {  // record the failure, then wait (bounded) for this warp's copies still in flight
    if (lane == 0 && a.err) atomicExch(a.err, 1);
    for (int j = ls; j < min(ls + NS, len); ++j) mbar_wait_bounded(&bars[j % NS], (uint32_t)((j / NS) & 1));
  }
  __syncthreads();
  l2_prefetch_share(a.pf, a.pf_bytes, blockIdx.x, gridDim.x);
  trace_mark(a.trace, 2);
}
#endif  // SSD_CROSSCHECK

// ---------------------------------------------------------------- batch-1 GEMV, register stream-K
//
// Equal slices of the (row pair, 1024-element chunk) steps for every warp of
// a grid of up to two CTAs per SM (gemv_warps: short rows get one warp per
// row pair, since splitting them finer costs more in merges than it gains;
// long rows are cut to about four slices per warp); a row pair cut by slice
// boundaries is merged by gemv_finish.  Each lane keeps its eight 16-byte
// weight loads of a step in registers (64 registers per thread): 16 warps per
// CTA and two CTAs per SM keep ~128 KB of loads in flight per SM.  Matrices
// with few row pairs run 2048-wide chunks instead (sixteen loads per lane,
// one CTA per SM), so a warp holding one row pair still has 8 KB in flight.  Before its
// dependency wait each warp prefetches the start of its slice into L2, 24 MB
// for the whole grid at most: under programmatic dependent launch the grid is
// resident while the previous kernel still streams its own weights, and a
// larger prefetch only takes HBM from it (or evicts itself from L2).  When a
// CTA has streamed its share it prefetches its share of the pass's next
// weight matrix into L2, so HBM stays busy across the kernel boundary.

constexpr int kRW = 16;  // warps per CTA

// Warps that share a matrix of nu row pairs and `total` (row pair, chunk)
// slices: one per row pair, or more when that leaves a warp more than four
// slices (long rows: the down projection's K = ffn).
__host__ __device__ __forceinline__ long long gemv_warps(int nu, long long total) {
  return nu > total / 4 ? (long long)nu : total / 4;
}

struct Pending {  // a warp's partial sums of a unit it shares with other warps
  int u, c0, c1;
  float y0, y1;
};

template <typename T, int CK>
__global__ void __launch_bounds__(512, CK == 1024 ? 2 : 1) k_gemv_rs(LinearArgs a) {
  constexpr int NL = CK / 256;  // 16-byte loads per lane and row for one chunk
  extern __shared__ __align__(16) float s_xr[];
  __shared__ float s_red[32];
  __shared__ Pending s_pend[kRW][2];
  griddep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = a.K;
  const int nu = n_units(a);
  const int nchunks = (K + CK - 1) / CK;
  const long long total = (long long)nu * nchunks;
  const int nw = (int)min((long long)gridDim.x * kRW, gemv_warps(nu, total));
  const int gw = blockIdx.x * kRW + warp;
  long long s0 = 0, s1 = 0;
  if (gw < nw) {
    s0 = total * gw / nw;
    s1 = total * (gw + 1) / nw;
  }
  const T* W = reinterpret_cast<const T*>(a.W);
  // Weights do not depend on the previous kernel: while it drains, pull the
  // first part of this warp's slice into L2 (unless a draft exit has already
  // closed this forward's gate: then the launch will do nothing).
  const bool warm = gate_open(a.gate);
  if (lane == 0 && warm) {
    size_t budget = min((size_t)64 * 1024, ((size_t)24 << 20) / (size_t)nw) & ~(size_t)31;
    for (long long s = s0; s < s1 && budget > 0;) {
      const int u = (int)(s / nchunks), c0 = (int)(s - (long long)u * nchunks);
      const int c1 = (int)min((long long)nchunks, c0 + (s1 - s));
      int r0, r1;
      unit_rows(a, u, r0, r1);
      const size_t e0 = (size_t)c0 * CK, e1 = min((size_t)c1 * CK, (size_t)K);
      size_t nb = (e1 - e0) * sizeof(T);
      if (nb > budget / 2) nb = (budget / 2) & ~(size_t)15;
      if (nb) {
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(W + (size_t)r0 * K + e0), "r"((uint32_t)nb)
                     : "memory");
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(W + (size_t)r1 * K + e0), "r"((uint32_t)nb)
                     : "memory");
      }
      budget = nb * 2 >= budget ? 0 : budget - nb * 2;
      s += c1 - c0;
    }
  }
  // The rest of the activation-independent work also goes before the wait: the RMSNorm gain into shared
  // memory and this warp's first weight step into registers.
  const T* G = reinterpret_cast<const T*>(a.gamma);
  T* s_g = reinterpret_cast<T*>(s_xr + K);
  if (G)  // each thread stages (and later reads) only its own elements
    for (int k = threadIdx.x * 8; k < K; k += blockDim.x * 8)
      *reinterpret_cast<uint4*>(s_g + k) = *reinterpret_cast<const uint4*>(G + k);
  uint4 q0[NL], q1[NL];
  auto load_step = [&](long long s) {
    const int u = (int)(s / nchunks), c = (int)(s - (long long)u * nchunks);
    int r0, r1;
    unit_rows(a, u, r0, r1);
    const int k0 = c * CK, n = min(CK, K - k0);
    const T* w0 = W + (size_t)r0 * K + k0;
    const T* w1 = W + (size_t)r1 * K + k0;
#pragma unroll
    for (int j = 0; j < NL; ++j) {
      const int e = lane * 8 + j * 256;
      if (e < n) {
        q0[j] = ld_stream16(w0 + e);
        q1[j] = ld_stream16(w1 + e);
      }
    }
  };
  if (warm && s0 < s1) load_step(s0);
  trace_mark(a.trace, 0);
  griddep_wait();
  if (!gate_open(a.gate)) return;
  if (!warm && s0 < s1) load_step(s0);
  trace_mark(a.trace, 1);

  // Activations: one pass from global into shared memory (sum of squares on the way), then RMSNorm /
  // int8 in place; every thread touches only its own elements, so only the reductions synchronise.
  float ss = 0.f;
  for (int k = threadIdx.x * 8; k < K; k += blockDim.x * 8) {
    const float4* xp = reinterpret_cast<const float4*>(a.X + k);
    const float4 u = xp[0], v = xp[1];
    float4* sp = reinterpret_cast<float4*>(s_xr + k);
    sp[0] = u;
    sp[1] = v;
    ss += u.x * u.x + u.y * u.y + u.z * u.z + u.w * u.w + v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  float inv = 1.0f;
  if (G) {
    ss = block_reduce(ss, s_red, false);
    inv = 1.0f / sqrtf(ss / (float)K + a.eps);
  }
  float qm = 0.f, qs = 0.f;
  if (a.int8) {
    float amax = 0.f;
    for (int k = threadIdx.x * 8; k < K; k += blockDim.x * 8) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float xv = s_xr[k + e];
        amax = fmaxf(amax, fabsf(G ? xv * inv * Io<T>::to_f(s_g[k + e]) : xv));
      }
    }
    amax = block_reduce(amax, s_red, true);
    if (amax > 0.f) {
      qm = __fdiv_rn(127.0f, amax);
      qs = __fdiv_rn(amax, 127.0f);
    }
  }
  if (G || a.int8) {
    for (int k = threadIdx.x * 8; k < K; k += blockDim.x * 8) {
      float4* sp = reinterpret_cast<float4*>(s_xr + k);
      const float4 u = sp[0], v = sp[1];
      float x[8] = {u.x, u.y, u.z, u.w, v.x, v.y, v.z, v.w};
      float g[8];
      if (G) Io<T>::unpack8(*reinterpret_cast<const uint4*>(s_g + k), g);
      prep8<T>(a, x, g, inv, qm);
      sp[0] = make_float4(x[0], x[1], x[2], x[3]);
      sp[1] = make_float4(x[4], x[5], x[6], x[7]);
    }
  }
  __syncthreads();
  float acc0 = 0.f, acc1 = 0.f;
  int npend = 0;
  for (long long s = s0; s < s1; ++s) {
    const int u = (int)(s / nchunks), c = (int)(s - (long long)u * nchunks);
    const int k0 = c * CK;
    const int n = min(CK, K - k0);
    if (s != s0) load_step(s);
#pragma unroll
    for (int j = 0; j < NL; ++j) {
      const int e = lane * 8 + j * 256;
      if (e < n) {
        float f0[8], f1[8];
        Io<T>::unpack8(q0[j], f0);
        Io<T>::unpack8(q1[j], f1);
        const float4* xp = reinterpret_cast<const float4*>(s_xr + k0 + e);
        const float4 xa = xp[0], xb = xp[1];
        const float x[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          acc0 = fmaf(f0[t], x[t], acc0);
          acc1 = fmaf(f1[t], x[t], acc1);
        }
      }
    }
    if (c == nchunks - 1 || s == s1 - 1) {
      const float y0 = warp_sum(acc0), y1 = warp_sum(acc1);
      acc0 = acc1 = 0.f;
      if (lane == 0) {
        const int c0 = (s - c) >= s0 ? 0 : (int)(s0 - (s - c));
        if (c0 == 0 && c == nchunks - 1) {
          epi_apply<T>(a, 0, u, a.int8 ? y0 * qs : y0, a.int8 ? y1 * qs : y1);
        } else {  // shared with other warps: only a slice's first and last unit can be
          if (npend < 2) s_pend[warp][npend++] = Pending{u, c0, c + 1, y0, y1};
        }
      }
    }
  }
  // merges of shared units, kept out of the streaming loop (its registers are spoken for)
  if (lane == 0)
    for (int i = 0; i < npend; ++i) {
      const Pending& pd = s_pend[warp][i];
      gemv_finish<T>(a, pd.u, pd.c0, pd.c1, nchunks, nw, pd.y0, pd.y1, qs);
    }
  __syncthreads();
  l2_prefetch_share(a.pf, a.pf_bytes, blockIdx.x, gridDim.x);
  trace_mark(a.trace, 2);
}

template <typename T>
static void run_gemv_rs(const LinearArgs& a, int sms, cudaStream_t st) {
  const int units = a.epi == EPI_SWIGLU ? a.F : a.N / 2;
  const size_t smem = (size_t)a.K * 4 + (a.gamma ? (size_t)a.K * sizeof(T) : 0);  // x, RMSNorm gain
  const int per_sm = smem <= 100 * 1024 ? 2 : 1;
  // also when the input row leaves room for one CTA per SM only (70B down projection, K = 28672): its 16 warps
  // then need the 2048-wide chunks' loads in flight, and a kernel built for two CTAs per SM whose CTAs take
  // 114 KB each moves the SM's carveout towards shared memory, leaving the GEMVs after it too little L1 for
  // their loads (70B draft pass 130.9 -> 94.7 ms: down 129.5 -> 72.9 us, gate/up 175 -> 138 us)
  if (units <= sms * kRW || per_sm == 1) {
    // matrices with no more row pairs than one CTA per SM has warps (the 8B O and down projections): one
    // warp per row pair with 1024-wide chunks leaves too few loads in flight; 2048-wide chunks (128
    // registers, one CTA per SM) double them per warp
    // One whole row pair per warp when that still keeps 80 % of the SMs streaming: no row pair is then split
    // between warps, so no partial sums are merged (8B down projection: 2048 row pairs on 128 CTAs, 23.4 ->
    // 19.5 us inside the draft graph, against 152 CTAs with split row pairs).
    const long long total = (long long)units * ((a.K + 2047) / 2048);
    const int whole = (units + kRW - 1) / kRW;
    const int grid = whole <= sms && 10 * whole >= 8 * sms
                         ? whole
                         : (int)std::min<long long>((gemv_warps(units, total) + kRW - 1) / kRW, (long long)sms);
    launch_ex(k_gemv_rs<T, 2048>, dim3(grid), dim3(kRW * 32), smem, st, a);
    return;
  }
  const long long total = (long long)units * ((a.K + kCK - 1) / kCK);
  int grid = (int)std::min<long long>((gemv_warps(units, total) + kRW - 1) / kRW, (long long)sms * per_sm);
  // Two CTAs per SM and at most 400 MB of weights: a grid that divides the row pairs, if one keeps at least
  // 80 % of the CTAs, so every CTA's slice starts and ends on a row-pair boundary and fewer row pairs are
  // merged (inside the draft graph: 8B gate/up on 256 instead of 304 CTAs 41.1 -> 38.6 us; 13B O, gate/up,
  // down, lm_head 15.6 / 63.1 / 34.1 / 71.2 -> 12.3 / 59.4 / 28.4 / 68.8 us).  Larger matrices keep the
  // uniform two-per-SM grid: their steady stream outweighs the tail (70B gate/up 175 us on 304 CTAs, 194 us
  // on 256).
  const size_t wbytes = (size_t)units * 2 * (size_t)a.K * sizeof(T);  // a unit is two weight rows
  if (per_sm == 2 && wbytes <= ((size_t)400 << 20))
    for (int g = grid; 10 * g >= 8 * grid; --g)
      if (units % g == 0) {
        grid = g;
        break;
      }
  launch_ex(k_gemv_rs<T, 1024>, dim3(grid), dim3(kRW * 32), smem, st, a);
}

void launch_gemv_rs(const LinearArgs& a, int fp16, int sms, cudaStream_t st) {
  if (fp16)
    run_gemv_rs<__half>(a, sms, st);
  else
    run_gemv_rs<__nv_bfloat16>(a, sms, st);
}

#ifdef SSD_CROSSCHECK
static size_t bulk_smem(int K, int ns, int elem) {
  return (((size_t)K * 4 + 127) & ~(size_t)127) + (size_t)kGW * ns * 2 * kCK * elem + (size_t)kGW * ns * 8;
}

constexpr int kBulkSmemMax = 220 * 1024;  // dynamic limit; the opt-in maximum also covers static shared memory

template <typename T>
static void run_gemv_bulk(const LinearArgs& a, int sms, cudaStream_t st) {
  const int units = a.epi == EPI_SWIGLU ? a.F : a.N / 2;
  int grid = (units + kGW - 1) / kGW;
  if (grid > sms) grid = sms;
  if (bulk_smem(a.K, 4, sizeof(T)) <= (size_t)kBulkSmemMax)
    launch_ex(k_gemv_bulk<T, 4>, dim3(grid), dim3(256), bulk_smem(a.K, 4, sizeof(T)), st, a);
  else
    launch_ex(k_gemv_bulk<T, 3>, dim3(grid), dim3(256), bulk_smem(a.K, 3, sizeof(T)), st, a);
}

void launch_gemv_bulk(const LinearArgs& a, int fp16, int sms, cudaStream_t st) {
  if (fp16)
    run_gemv_bulk<__half>(a, sms, st);
  else
    run_gemv_bulk<__nv_bfloat16>(a, sms, st);
}
#endif  // SSD_CROSSCHECK

bool init_linear_kernels() {
  bool ok = true;
#ifdef SSD_CROSSCHECK
  const int mx = kBulkSmemMax;
  ok &= cudaFuncSetAttribute(k_gemv_bulk<__half, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx) == cudaSuccess;
  ok &= cudaFuncSetAttribute(k_gemv_bulk<__half, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx) == cudaSuccess;
  ok &= cudaFuncSetAttribute(k_gemv_bulk<__nv_bfloat16, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx) ==
        cudaSuccess;
  ok &= cudaFuncSetAttribute(k_gemv_bulk<__nv_bfloat16, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx) ==
        cudaSuccess;
  ok &= cudaFuncSetAttribute(k_gemv<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024) == cudaSuccess;
  ok &= cudaFuncSetAttribute(k_gemv<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024) ==
        cudaSuccess;
#endif
  ok &= cudaFuncSetAttribute(k_gemv_rs<__half, 1024>, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024) ==
        cudaSuccess;
  ok &= cudaFuncSetAttribute(k_gemv_rs<__nv_bfloat16, 1024>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             160 * 1024) == cudaSuccess;
  ok &= cudaFuncSetAttribute(k_gemv_rs<__half, 2048>, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024) ==
        cudaSuccess;
  ok &= cudaFuncSetAttribute(k_gemv_rs<__nv_bfloat16, 2048>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             160 * 1024) == cudaSuccess;
  return ok;
}

#ifdef SSD_CROSSCHECK
void launch_gemv(const LinearArgs& a, int fp16, cudaStream_t st) {
  if (fp16)
    run_gemv<__half>(a, st);
  else
    run_gemv<__nv_bfloat16>(a, st);
}
#endif  // SSD_CROSSCHECK

}  // namespace ssd

extern "C" int64_t ssd_gemv_warps(int nu, int64_t total) { return ssd::gemv_warps(nu, total); }
