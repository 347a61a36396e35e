// Decode / verify / tree / CLaSp-DP attention over the paged KV cache.
//
// Row r sees cache slots [0, prefix) and the new slots base + e for every bit
// e of mask[r] (PassDesc).  The same kernel serves linear drafts, the
// causal verify of K+1 rows, the tree-masked verify (mask = ancestors), the
// DP rows (mask = own slot; prefix = the target's position) and prefill
// chunks.  Keys are indexed 0..prefix-1 (prefix) then prefix..prefix+63
// (new slots); the key range is split across CTAs, each CTA keeps an online
// softmax (running max m, sum l, weighted V sum) per query, and the last CTA
// of a (kv head, query block) merges the splits.  All query heads of a GQA
// group and all rows read each K/V tile once.
#include <cooperative_groups.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace ssd {

constexpr int kTile = 32;  // keys per shared-memory tile (one per lane)
constexpr int kQB = 16;    // queries per CTA (4 warps x 4)

int attention_qblocks(int rows, int group) { return (rows * group + kQB - 1) / kQB; }

// Eight consecutive cache elements as fp32 (16-bit caches: one 16-byte load).
template <typename CT>
__device__ __forceinline__ void load8(const CT* p, float out[8]) {
  Io<CT>::unpack8(*reinterpret_cast<const uint4*>(p), out);
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, float out[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  out[0] = a.x;
  out[1] = a.y;
  out[2] = a.z;
  out[3] = a.w;
  out[4] = b.x;
  out[5] = b.y;
  out[6] = b.z;
  out[7] = b.w;
}

template <typename T, int HD>
__global__ void __launch_bounds__(128) k_attention(AttnArgs a) {
  constexpr int DPL = HD / 32;  // output dims per lane
  __shared__ float s_k[kTile][HD + 1];
  __shared__ float s_v[kTile][HD + 1];
  __shared__ float s_q[kQB][HD];
  __shared__ float s_p[4][4][kTile];

  griddep_launch();
  // the next projection's weights do not depend on any predecessor: start their L2 prefetch now
  l2_prefetch_share(a.pf, a.pf_bytes, (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x,
                    gridDim.x * gridDim.y * gridDim.z);
  trace_mark(a.trace, 0);
  griddep_wait();
  trace_mark(a.trace, 1);
  const PassDesc* d = a.desc;
  const int kvh = blockIdx.x, split = blockIdx.y, qblk = blockIdx.z;
  const int group = a.n_q / a.n_kv;
  const int nq = a.rows * group;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int prefix = d->prefix, base = d->base;
  const int total = prefix + a.rows;
  const int chunk = (total + a.n_split - 1) / a.n_split;
  const int k0 = split * chunk, k1 = min(total, k0 + chunk);
  const float scale = rsqrtf((float)HD);

  // queries of this CTA: index qi = r * group + g  ->  row r, head kvh*group + g (float4 loads)
  constexpr int QV = kQB * HD / 4 / 128;  // float4 per thread
#pragma unroll
  for (int it = 0; it < QV; ++it) {
    const int i = (it * 128 + threadIdx.x) * 4;
    const int ql = i / HD, dd = i - ql * HD;
    const int qi = qblk * kQB + ql;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (qi < nq) {
      const int r = qi / group, h = kvh * group + (qi - r * group);
      v = *reinterpret_cast<const float4*>(a.q + (size_t)r * a.n_q * HD + h * HD + dd);
      v.x *= scale;
      v.y *= scale;
      v.z *= scale;
      v.w *= scale;
    }
    *reinterpret_cast<float4*>(&s_q[ql][dd]) = v;
  }

  float m_run[4], l_run[4], acc[4][DPL];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    m_run[j] = -INFINITY;
    l_run[j] = 0.f;
#pragma unroll
    for (int c = 0; c < DPL; ++c) acc[j][c] = 0.f;
  }
  const T* kc = reinterpret_cast<const T*>(a.kcache);
  const T* vc = reinterpret_cast<const T*>(a.vcache);
  bool qvalid[4];
  unsigned long long qmask[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int qi = qblk * kQB + warp * 4 + j;
    qvalid[j] = qi < nq;
    qmask[j] = qvalid[j] ? d->mask[qi / group] : 0ull;
  }

  // K/V tiles: every thread holds TL 16-byte chunks of K and of V; the next
  // tile's loads are issued before the current tile is computed.
  constexpr int TL = kTile * (HD / 8) / 128;
  float kr[TL][8], vr[TL][8];
  auto load_tile = [&](int t0) {
#pragma unroll
    for (int it = 0; it < TL; ++it) {
      const int i = it * 128 + threadIdx.x;
      const int kk = i / (HD / 8), dd = (i - kk * (HD / 8)) * 8;
      const int key = t0 + kk;
      if (key < k1) {
        const int slot = key < prefix ? key : base + (key - prefix);
        const size_t idx = kv_index(a.layer, slot, kvh, dd, a.btab, a.n_pages, a.n_kv, HD);
        load8<T>(kc + idx, kr[it]);
        load8<T>(vc + idx, vr[it]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) kr[it][e] = vr[it][e] = 0.f;
      }
    }
  };
  if (k0 < k1) load_tile(k0);
  for (int t0 = k0; t0 < k1; t0 += kTile) {
    __syncthreads();
#pragma unroll
    for (int it = 0; it < TL; ++it) {
      const int i = it * 128 + threadIdx.x;
      const int kk = i / (HD / 8), dd = (i - kk * (HD / 8)) * 8;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        s_k[kk][dd + e] = kr[it][e];
        s_v[kk][dd + e] = vr[it][e];
      }
    }
    if (t0 + kTile < k1) load_tile(t0 + kTile);
    __syncthreads();
    if (qblk * kQB + warp * 4 >= nq) continue;  // no query in this warp (warp-uniform)
    // the warp's four queries together: lane = key of the tile
    const int key = t0 + lane;
    float dot[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int dd = 0; dd < HD; ++dd) {
      const float kv = s_k[lane][dd];
#pragma unroll
      for (int j = 0; j < 4; ++j) dot[j] = fmaf(s_q[warp * 4 + j][dd], kv, dot[j]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool vis = qvalid[j] && key < k1 && (key < prefix || ((qmask[j] >> (key - prefix)) & 1ull));
      const float sc = vis ? dot[j] : -INFINITY;
      const float tmax = warp_max(sc);
      float p = 0.f;
      if (tmax != -INFINITY) {
        const float m_new = fmaxf(m_run[j], tmax);
        const float corr = expf(m_run[j] - m_new);  // exp(-inf) = 0 on the first visible tile
        p = vis ? expf(sc - m_new) : 0.f;
        l_run[j] = l_run[j] * corr + warp_sum(p);
#pragma unroll
        for (int c = 0; c < DPL; ++c) acc[j][c] *= corr;
        m_run[j] = m_new;
      }
      s_p[warp][j][lane] = p;
    }
    __syncwarp();
#pragma unroll 4
    for (int kk = 0; kk < kTile; ++kk) {
      float v[DPL];
#pragma unroll
      for (int c = 0; c < DPL; ++c) v[c] = s_v[kk][lane + 32 * c];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float pj = s_p[warp][j][kk];
#pragma unroll
        for (int c = 0; c < DPL; ++c) acc[j][c] = fmaf(pj, v[c], acc[j][c]);
      }
    }
    __syncwarp();
  }

  // Merge across the splits of this (kv head, query block): the splits form
  // one thread-block cluster; each CTA leaves its partial softmax states
  // (m, l, weighted V sum) in its own shared memory (the K tile buffer is
  // free now) and the ranks merge disjoint queries over distributed shared
  // memory -- no global partials, fences or arrival counters.
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  constexpr int PS = HD + 2;
  __syncthreads();
  float* s_part = &s_k[0][0];  // [kQB][HD + 2]
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int ql = warp * 4 + j;
    if (lane == 0) {
      s_part[ql * PS] = m_run[j];
      s_part[ql * PS + 1] = l_run[j];
    }
#pragma unroll
    for (int c = 0; c < DPL; ++c) s_part[ql * PS + 2 + lane + 32 * c] = acc[j][c];
  }
  cluster.sync();
  const int nsp = (int)cluster.num_blocks(), rank = (int)cluster.block_rank();
  for (int t = warp; rank + nsp * t < kQB; t += 4) {
    const int ql = rank + nsp * t;
    const int qi = qblk * kQB + ql;
    if (qi >= nq) continue;
    float ms = -INFINITY, lsum = 0.f;
    if (lane < nsp) {
      const float* rp = cluster.map_shared_rank(s_part, (unsigned)lane);
      ms = rp[ql * PS];
      lsum = rp[ql * PS + 1];
    }
    const float M = warp_max(ms);
    const float w = (ms == -INFINITY) ? 0.f : expf(ms - M);
    const float L = warp_sum(lsum * w);
    float o[DPL];
#pragma unroll
    for (int c = 0; c < DPL; ++c) o[c] = 0.f;
    for (int sp = 0; sp < nsp; ++sp) {
      const float ws = __shfl_sync(0xffffffffu, w, sp);
      const float* rp = cluster.map_shared_rank(s_part, (unsigned)sp) + ql * PS + 2;
#pragma unroll
      for (int c = 0; c < DPL; ++c) o[c] = fmaf(ws, rp[lane + 32 * c], o[c]);
    }
    const int r = qi / group, h = kvh * group + (qi - r * group);
    float* out = a.out + (size_t)r * a.n_q * HD + h * HD;
    const float invL = L > 0.f ? 1.0f / L : 0.f;
#pragma unroll
    for (int c = 0; c < DPL; ++c) out[lane + 32 * c] = o[c] * invL;
  }
  cluster.sync();  // every CTA's shared memory stays alive until all ranks have read it
  trace_mark(a.trace, 2);
}

int attention_splits(int max_keys) {
  if (max_keys <= 64) return 1;
  if (max_keys <= 128) return 2;
  if (max_keys <= 256) return 4;
  return 8;
}

template <typename T>
static void run_attn(const AttnArgs& a, cudaStream_t st) {
  const int group = a.n_q / a.n_kv;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;  // the splits of one (kv head, query block)
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = a.n_split;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(a.n_kv, a.n_split, attention_qblocks(a.rows, group));
  cfg.blockDim = dim3(128);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = g_pdl ? 2 : 1;
  g_launches += 1;
  if (a.hd == 128)
    cudaLaunchKernelEx(&cfg, k_attention<T, 128>, a);
  else
    cudaLaunchKernelEx(&cfg, k_attention<T, 64>, a);
}

void launch_attention(const AttnArgs& a, int kv_type, cudaStream_t st) {
  if (kv_type == 2)
    run_attn<float>(a, st);
  else if (kv_type == 1)
    run_attn<__half>(a, st);
  else
    run_attn<__nv_bfloat16>(a, st);
}

}  // namespace ssd
