// Decode / verify / tree / CLaSp-DP attention over the paged KV cache.
//
// Row r sees cache slots [0, prefix) and the new slots base + e for every bit
// e of mask[r] (PassDesc).  The same kernel serves linear drafts, the
// causal verify of K+1 rows, the tree-masked verify (mask = ancestors), the
// DP rows (mask = own slot; prefix = the target's position) and prefill
// chunks.
//
// Keys are cut into tiles of 32: ceil(prefix / 32) prefix tiles (each inside
// one 64-slot page, so one (page, kv head) block of rows) and ceil(rows / 32)
// tiles of new slots.  A (kv head, query block) is a thread-block cluster of
// n_split CTAs; each CTA takes a contiguous run of tiles.  Prefix tiles come
// in by TMA (2D tensor map over one layer of the cache, 128-byte swizzle, so
// that a lane reading its own key's row and a lane reading its own dims of
// a row are both free of bank conflicts); new-slot tiles (written by the
// projection just before) by plain loads into the same layout.  Before its
// dependency wait each CTA prefetches its prefix tiles into L2, so the cache
// reads overlap the end of the QKV projection.
//
// Each warp owns four queries; when a CTA has fewer than 16 queries (decode:
// one row x the GQA group), the warps that share a query group split the
// tiles instead.  Every warp keeps an online softmax (running max m, sum l,
// weighted V sum) per query; the partial states of all warps of all CTAs
// of the cluster are merged over distributed shared memory in a fixed order.
#include <cooperative_groups.h>
#include <cuda.h>
#include <math.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace ssd {

constexpr int kTile = 32;                    // keys per tile (one per lane in Q.K)
constexpr int kQB = 16;                      // queries per CTA (4 warps x 4)
constexpr int kMaxSlots = 8;                 // tiles held in shared memory at once
constexpr int kRingBudget = 192 * 1024;      // shared memory for the tile ring
constexpr int kBoxBytes = kTile * 128;       // one TMA box: 32 rows x 128 bytes

int attention_qblocks(int rows, int group) { return (rows * group + kQB - 1) / kQB; }

template <typename T, int HD>
struct TileGeo {
  static constexpr int kRowBytes = HD * (int)sizeof(T);
  static constexpr int kBoxes = kRowBytes / 128;      // 128-byte column boxes per row
  static constexpr int kHalf = kBoxes * kBoxBytes;    // K (or V) of one tile
  static constexpr int kSlot = 2 * kHalf;             // K then V
  static constexpr int kSlots = kRingBudget / kSlot < kMaxSlots ? kRingBudget / kSlot : kMaxSlots;
  static constexpr int kChunk = 16 / (int)sizeof(T);  // elements per 16-byte chunk
  static constexpr int kChunks = HD / kChunk;         // 16-byte chunks per row
};

// Byte offset of byte x of tile row r in the swizzled layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B: 16-byte chunk c of a 128-byte line moves to c ^ (r % 8).
__device__ __forceinline__ int swz(int r, int x) {
  return (x >> 7) * kBoxBytes + r * 128 + ((((x >> 4) & 7) ^ (r & 7)) << 4) + (x & 15);
}

template <typename T>
__device__ __forceinline__ void unpack16(const uint4& u, float* f);
template <>
__device__ __forceinline__ void unpack16<float>(const uint4& u, float* f) {
  f[0] = __uint_as_float(u.x);
  f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z);
  f[3] = __uint_as_float(u.w);
}
template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4& u, float* f) {
  Io<__nv_bfloat16>::unpack8(u, f);
}
template <>
__device__ __forceinline__ void unpack16<__half>(const uint4& u, float* f) {
  Io<__half>::unpack8(u, f);
}

__device__ __forceinline__ float2 to_float2(__half2 h) { return __half22float2(h); }
__device__ __forceinline__ float2 to_float2(__nv_bfloat162 h) { return __bfloat1622float2(h); }

// N consecutive elements (N * sizeof(T) in {4, 8, 16} bytes, naturally aligned) as fp32.
template <typename T, int N>
__device__ __forceinline__ void lds_elems(const unsigned char* p, float* f) {
  if constexpr (sizeof(T) == 4) {
    if constexpr (N == 4) {
      const float4 v = *reinterpret_cast<const float4*>(p);
      f[0] = v.x, f[1] = v.y, f[2] = v.z, f[3] = v.w;
    } else {
      const float2 v = *reinterpret_cast<const float2*>(p);
      f[0] = v.x, f[1] = v.y;
    }
  } else {
    using H2 = typename std::conditional<std::is_same<T, __half>::value, __half2, __nv_bfloat162>::type;
    if constexpr (N == 4) {
      const uint2 u = *reinterpret_cast<const uint2*>(p);
      const H2 a = *reinterpret_cast<const H2*>(&u.x), b = *reinterpret_cast<const H2*>(&u.y);
      const float2 fa = to_float2(a), fb = to_float2(b);
      f[0] = fa.x, f[1] = fa.y, f[2] = fb.x, f[3] = fb.y;
    } else {
      const H2 a = *reinterpret_cast<const H2*>(p);
      const float2 fa = to_float2(a);
      f[0] = fa.x, f[1] = fa.y;
    }
  }
}

__device__ __forceinline__ void tma_load_rows(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void l2_prefetch(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Tiles [t0, t1) of split `split` out of n_tiles over ns splits.
__device__ __forceinline__ void split_tiles(int n_tiles, int split, int ns, int& t0, int& t1) {
  t0 = (int)((long long)n_tiles * split / ns);
  t1 = (int)((long long)n_tiles * (split + 1) / ns);
}

template <typename T, int HD>
__global__ void __launch_bounds__(128) k_attention(const __grid_constant__ CUtensorMap tk,
                                                   const __grid_constant__ CUtensorMap tv, AttnArgs a) {
  using G = TileGeo<T, HD>;
  constexpr int DPL = HD / 32;  // output dims per lane (lane owns dims lane*DPL ..)
  constexpr int PS = HD + 2;    // partial state: m, l, weighted V sum
  extern __shared__ unsigned char s_dyn[];
  __shared__ __align__(16) float s_q[kQB][HD];
  __shared__ float s_p[4][4][kTile];
  __shared__ float s_part[4][4][PS];
  __shared__ __align__(8) uint64_t s_full[kMaxSlots];
  __shared__ int s_fail;
  unsigned char* ring =
      s_dyn + ((1024 - (smem_u32(s_dyn) & 1023)) & 1023);  // SWIZZLE_128B wants 1024-byte aligned boxes

  const int kvh = blockIdx.x, split = blockIdx.y, qblk = blockIdx.z, ns = gridDim.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.n_slots;
  const size_t layer_rows = (size_t)a.n_pages * a.n_kv * kPage;
  const T* kc = reinterpret_cast<const T*>(a.kcache) + (size_t)a.layer * layer_rows * HD;
  const T* vc = reinterpret_cast<const T*>(a.vcache) + (size_t)a.layer * layer_rows * HD;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) mbar_init(&s_full[i], 1);
    fence_barrier_init();
    s_fail = 0;
  }

  griddep_launch();
  // An L2 prefetch only warms the cache, so it may run before the wait: this CTA's prefix tiles, found
  // through the block table (never written on the device).  The descriptor may still hold the previous
  // pass's prefix (each pass rewrites it at its start); that only makes the prefetch slightly off, never
  // out of range.
  {
    const int hint = min(*reinterpret_cast<const volatile int*>(&a.desc->prefix), a.n_pages * kPage);
    const int pt = (hint + kTile - 1) / kTile;
    int t0, t1;
    split_tiles(pt + (a.rows + kTile - 1) / kTile, split, ns, t0, t1);
    t1 = min(t1, pt);
    for (int i = threadIdx.x; i < 2 * (t1 - t0); i += blockDim.x) {
      const int ti = t0 + (i >> 1), key = ti * kTile;
      const size_t row = ((size_t)a.btab[key / kPage] * a.n_kv + kvh) * kPage + (key % kPage);
      l2_prefetch(((i & 1) ? vc : kc) + row * HD, (uint32_t)(kTile * G::kRowBytes));
    }
  }
  l2_prefetch_share(a.pf, a.pf_bytes, (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x,
                    gridDim.x * gridDim.y * gridDim.z);
  trace_mark(a.trace, 0);
  griddep_wait();
  trace_mark(a.trace, 1);

  const PassDesc* d = a.desc;
  const int group = a.n_q / a.n_kv;
  const int nq = a.rows * group;
  const int prefix = d->prefix, base = d->base;
  const int pt = (prefix + kTile - 1) / kTile;
  int tb, te;
  split_tiles(pt + (a.rows + kTile - 1) / kTile, split, ns, tb, te);
  const float scale = rsqrtf((float)HD);

  // queries of this CTA: index qi = r * group + g  ->  row r, head kvh*group + g
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

  // warp roles: query group wq (4 queries), tile share wk of WK
  const int nqc = min(kQB, nq - qblk * kQB);
  const int WQ = nqc <= 4 ? 1 : (nqc <= 8 ? 2 : 4);
  const int WK = 4 / WQ;
  const int wq = warp % WQ, wk = warp / WQ;
  float m_run[4], l_run[4], acc[4][DPL];
  bool qvalid[4];
  unsigned long long qmask[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    m_run[j] = -INFINITY;
    l_run[j] = 0.f;
#pragma unroll
    for (int c = 0; c < DPL; ++c) acc[j][c] = 0.f;
    const int qi = qblk * kQB + wq * 4 + j;
    qvalid[j] = qi < nq;
    qmask[j] = qvalid[j] ? d->mask[qi / group] : 0ull;
  }
  const float* sq = &s_q[wq * 4][0];
  bool ok = true;

  for (int b0 = tb; b0 < te; b0 += S) {
    const int nb = min(S, te - b0);
    const uint32_t phase = (uint32_t)((b0 - tb) / S) & 1u;
    if (threadIdx.x == 0) {
      fence_proxy_async();  // the previous batch's reads of the ring come before these async-proxy writes
      for (int i = 0; i < nb && b0 + i < pt; ++i) {
        const int key = (b0 + i) * kTile;
        const int row = (a.btab[key / kPage] * a.n_kv + kvh) * kPage + (key % kPage);
        unsigned char* slot = ring + (size_t)i * G::kSlot;
        mbar_expect_tx(&s_full[i], (uint32_t)G::kSlot);
#pragma unroll
        for (int bx = 0; bx < G::kBoxes; ++bx) {
          tma_load_rows(slot + bx * kBoxBytes, &tk, bx * (128 / (int)sizeof(T)), row, &s_full[i]);
          tma_load_rows(slot + G::kHalf + bx * kBoxBytes, &tv, bx * (128 / (int)sizeof(T)), row, &s_full[i]);
        }
      }
    }
    // tiles of new slots: plain 16-byte loads into the same swizzled layout (zeros past the last row)
    for (int i = max(0, pt - b0); i < nb; ++i) {
      const int e0 = (b0 + i - pt) * kTile;
      unsigned char* slot = ring + (size_t)i * G::kSlot;
      for (int idx = threadIdx.x; idx < kTile * G::kChunks; idx += blockDim.x) {
        const int r = idx / G::kChunks, c = idx - r * G::kChunks;
        const int e = e0 + r;
        uint4 kq = make_uint4(0, 0, 0, 0), vq = kq;
        if (e < a.rows) {
          const size_t gi = kv_index(a.layer, base + e, kvh, c * G::kChunk, a.btab, a.n_pages, a.n_kv, HD);
          kq = *reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(a.kcache) + gi);
          vq = *reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(a.vcache) + gi);
        }
        *reinterpret_cast<uint4*>(slot + swz(r, c * 16)) = kq;
        *reinterpret_cast<uint4*>(slot + G::kHalf + swz(r, c * 16)) = vq;
      }
    }
    __syncthreads();

    for (int i = wk; i < nb; i += WK) {
      const int ti = b0 + i;
      const bool is_prefix = ti < pt;
      if (is_prefix && !mbar_wait_bounded(&s_full[i], phase)) {
        ok = false;  // record it, give the copies in flight one more bounded wait, issue no more
        mbar_wait_bounded(&s_full[i], phase);
        s_fail = 1;
        continue;
      }
      const int k0 = is_prefix ? ti * kTile : (ti - pt) * kTile;  // first key (prefix) or new-slot index
      const int nvalid = is_prefix ? min(kTile, prefix - k0) : min(kTile, a.rows - k0);
      const unsigned char* kt = ring + (size_t)i * G::kSlot;
      const unsigned char* vt = kt + G::kHalf;

      // scores: lane = key of the tile
      float dot[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
      for (int c = 0; c < G::kChunks; ++c) {
        const uint4 raw = *reinterpret_cast<const uint4*>(kt + swz(lane, c * 16));
        float kf[G::kChunk];
        unpack16<T>(raw, kf);
#pragma unroll
        for (int h = 0; h < G::kChunk; h += 4) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float4 qv = *reinterpret_cast<const float4*>(sq + j * HD + c * G::kChunk + h);
            dot[j] = fmaf(qv.x, kf[h], dot[j]);
            dot[j] = fmaf(qv.y, kf[h + 1], dot[j]);
            dot[j] = fmaf(qv.z, kf[h + 2], dot[j]);
            dot[j] = fmaf(qv.w, kf[h + 3], dot[j]);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool vis = qvalid[j] && lane < nvalid && (is_prefix || ((qmask[j] >> (k0 + lane)) & 1ull));
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
      // weighted V sum: lane = dims lane*DPL ..; rows past nvalid are never read
      const int xb = lane * DPL * (int)sizeof(T);
#pragma unroll 4
      for (int kk = 0; kk < nvalid; ++kk) {
        float v[DPL];
        lds_elems<T, DPL>(vt + swz(kk, xb), v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float pj = s_p[warp][j][kk];
#pragma unroll
          for (int c = 0; c < DPL; ++c) acc[j][c] = fmaf(pj, v[c], acc[j][c]);
        }
      }
      __syncwarp();
    }
    __syncthreads();  // the ring is reused by the next batch
    if (s_fail) break;
  }
  if (!ok && lane == 0 && a.err) atomicExch(a.err, 1);

  // Partial states of this warp's queries, then the merge over all warps of
  // all CTAs of the cluster (distributed shared memory), queries spread over
  // the ranks; the order of the sum is fixed.
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (lane == 0) {
      s_part[warp][j][0] = m_run[j];
      s_part[warp][j][1] = l_run[j];
    }
#pragma unroll
    for (int c = 0; c < DPL; ++c) s_part[warp][j][2 + lane * DPL + c] = acc[j][c];
  }
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  const int nsp = (int)cluster.num_blocks(), rank = (int)cluster.block_rank();
  const int nst = nsp * WK;  // partial states per query (<= 32)
  for (int t = warp; rank + nsp * t < kQB; t += 4) {
    const int ql = rank + nsp * t;
    const int qi = qblk * kQB + ql;
    if (qi >= nq) continue;
    const int qg = ql >> 2, j = ql & 3;
    float ms = -INFINITY, lsum = 0.f;
    if (lane < nst) {
      const float* rp = cluster.map_shared_rank(&s_part[qg + WQ * (lane % WK)][j][0], (unsigned)(lane / WK));
      ms = rp[0];
      lsum = rp[1];
    }
    const float M = warp_max(ms);
    const float w = (ms == -INFINITY) ? 0.f : expf(ms - M);
    const float L = warp_sum(lsum * w);
    float o[DPL];
#pragma unroll
    for (int c = 0; c < DPL; ++c) o[c] = 0.f;
    for (int sidx = 0; sidx < nst; ++sidx) {
      const float ws = __shfl_sync(0xffffffffu, w, sidx);
      const float* rp = cluster.map_shared_rank(&s_part[qg + WQ * (sidx % WK)][j][0], (unsigned)(sidx / WK));
#pragma unroll
      for (int c = 0; c < DPL; ++c) o[c] = fmaf(ws, rp[2 + lane * DPL + c], o[c]);
    }
    const int r = qi / group, h = kvh * group + (qi - r * group);
    float* out = a.out + (size_t)r * a.n_q * HD + h * HD + lane * DPL;
    const float invL = L > 0.f ? 1.0f / L : 0.f;
#pragma unroll
    for (int c = 0; c < DPL; ++c) out[c] = o[c] * invL;
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

namespace {

template <typename T, int HD>
constexpr size_t attn_smem(int slots) {
  return 1024 + (size_t)slots * TileGeo<T, HD>::kSlot;
}

template <typename T, int HD>
bool set_attn_attr() {
  return cudaFuncSetAttribute(k_attention<T, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)attn_smem<T, HD>(TileGeo<T, HD>::kSlots)) == cudaSuccess;
}

bool attn_attrs() {
  static std::once_flag once;
  static bool ok = false;
  std::call_once(once, [] {
    ok = set_attn_attr<float, 64>() && set_attn_attr<float, 128>() && set_attn_attr<__half, 64>() &&
         set_attn_attr<__half, 128>() && set_attn_attr<__nv_bfloat16, 64>() && set_attn_attr<__nv_bfloat16, 128>();
  });
  return ok;
}

template <typename T, int HD>
bool run_attn(const AttnArgs& in, cudaStream_t st) {
  using G = TileGeo<T, HD>;
  if (!attn_attrs()) return false;
  AttnArgs a = in;
  // one layer of the cache as a [rows][HD] matrix, boxes of 32 rows x 128 bytes
  const uint64_t layer_rows = (uint64_t)a.n_pages * a.n_kv * kPage;
  const size_t layer_elems = (size_t)layer_rows * HD;
  const CUtensorMapDataType dt = sizeof(T) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  CUtensorMap tk, tv;
  if (!encode_rows_2d(&tk, reinterpret_cast<const T*>(a.kcache) + (size_t)a.layer * layer_elems, dt, sizeof(T), HD,
                      layer_rows, 128 / sizeof(T), kTile) ||
      !encode_rows_2d(&tv, reinterpret_cast<const T*>(a.vcache) + (size_t)a.layer * layer_elems, dt, sizeof(T), HD,
                      layer_rows, 128 / sizeof(T), kTile))
    return false;
  // ring slots: the most tiles one split can get, capped by the shared-memory budget
  const int max_tiles = (a.max_keys + kTile - 1) / kTile + 1;
  a.n_slots = std::max(1, std::min(G::kSlots, (max_tiles + a.n_split - 1) / a.n_split));
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
  cfg.dynamicSmemBytes = attn_smem<T, HD>(a.n_slots);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = g_pdl ? 2 : 1;
  g_launches += 1;
  return cudaLaunchKernelEx(&cfg, k_attention<T, HD>, tk, tv, a) == cudaSuccess;
}

template <typename T>
bool run_attn_hd(const AttnArgs& a, cudaStream_t st) {
  return a.hd == 128 ? run_attn<T, 128>(a, st) : run_attn<T, 64>(a, st);
}

}  // namespace

bool init_attention_kernels() { return attn_attrs(); }

bool launch_attention(const AttnArgs& a, int kv_type, cudaStream_t st) {
  if (a.n_split < 1 || a.n_split > 8 || a.rows < 1 || a.rows > kMaxRows || (a.hd != 64 && a.hd != 128)) return false;
  if (((uintptr_t)a.kcache | (uintptr_t)a.vcache) & 15) return false;  // TMA wants 16-byte aligned tensors
  if (kv_type == 2) return run_attn_hd<float>(a, st);
  if (kv_type == 1) return run_attn_hd<__half>(a, st);
  return run_attn_hd<__nv_bfloat16>(a, st);
}

}  // namespace ssd
