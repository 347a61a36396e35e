// Decode / verify / tree / CLaSp-DP attention over the paged KV cache.
//
// Row r sees cache slots [0, prefix) and the new slots base + e for every bit
// e of mask[r] (PassDesc).  The same kernel serves linear drafts, the
// causal verify of K+1 rows, the tree-masked verify (mask = ancestors), the
// DP rows (mask = own slot; prefix = the target's position) and prefill
// chunks.
//
// Keys are cut into tiles of 32, each inside one 64-slot page (one (page, kv
// head) block of rows).  When the new slots continue the prefix (base ==
// prefix: every pass but the DP's) the keys [0, prefix + rows) are tiled
// together; otherwise ceil(prefix / 32) prefix tiles are followed by
// ceil(rows / 32) tiles of new slots.  A (kv head, query block) is a
// thread-block cluster of n_split CTAs; each CTA takes a contiguous run of
// tiles.  Tiles come in by TMA (2D tensor map over one layer of the cache,
// 128-byte swizzle, so that a lane reading its own key's row and a lane
// reading its own dims of a row are both free of bank conflicts); separately
// tiled new slots (written by the projection just before, anywhere in their
// pages) by plain loads into the same layout.  Before its dependency wait
// each CTA prefetches its prefix tiles into L2 and, in graph-replayed
// passes, copies the first ones into its ring, so the cache reads overlap
// the end of the QKV projection.
//
// A CTA holds a block of qb (4 to 32) queries in groups of four (of one when
// the block holds at most four queries) and runs 16 warps: each warp owns one
// query group, and the warps that share a group split the tiles between
// them.  The query-block size and the split count are chosen per launch
// shape (attention_layout).  Tiles pass through a ring
// of shared-memory slots; when a CTA has more tiles than slots, every tile
// of a slot goes to the warps that released the tile before it (the slot's
// mbarrier waits only tell consecutive phases apart).  Every warp keeps an
// online softmax (running max m, sum l, weighted V sum) per query; the
// partial states of all warps of all CTAs of the cluster are merged over
// distributed shared memory in a fixed order.
#include <cooperative_groups.h>
#include <cuda.h>
#include <math.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace ssd {

constexpr int kTile = 32;                // keys per tile (one per lane in Q.K)
constexpr int kWarps = 16;              // warps per CTA
constexpr int kQB = 32;                 // most queries per CTA (eight groups of four)
constexpr int kMaxSlots = 8;            // tiles held in shared memory at once
constexpr int kRingBudget = 192 * 1024; // shared memory for the tile ring
constexpr int kBoxBytes = kTile * 128;  // one TMA box: 32 rows x 128 bytes


template <typename T, int HD>
struct TileGeo {
  static constexpr int kRowBytes = HD * (int)sizeof(T);
  static constexpr int kBoxes = kRowBytes / 128;      // 128-byte column boxes per row
  static constexpr int kHalf = kBoxes * kBoxBytes;    // K (or V) of one tile
  static constexpr int kSlot = 2 * kHalf;             // K then V
  static constexpr int kSlots = kRingBudget / kSlot < kMaxSlots ? kRingBudget / kSlot : kMaxSlots;
  static constexpr int kChunk = 16 / (int)sizeof(T);  // elements per 16-byte chunk
  static constexpr int kChunks = HD / kChunk;         // 16-byte chunks per row
  static constexpr int kPartBytes = (kWarps * 4 + kQB) * (HD + 4) * 4;  // per-warp and per-CTA partial states
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

// 16-byte global -> shared copy that bypasses L1.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
// Arrive on bar once this thread's earlier cp.async copies have landed (not one of the expected arrivals).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// N consecutive floats (N = 2 or 4, 8- or 16-byte aligned; shared, distributed shared or global memory).
template <int N>
__device__ __forceinline__ void load_dims(const float* p, float* v) {
  if constexpr (N == 4) {
    const float4 t = *reinterpret_cast<const float4*>(p);
    v[0] = t.x, v[1] = t.y, v[2] = t.z, v[3] = t.w;
  } else {
    const float2 t = *reinterpret_cast<const float2*>(p);
    v[0] = t.x, v[1] = t.y;
  }
}
template <int N>
__device__ __forceinline__ void store_dims(float* p, const float* v) {
  if constexpr (N == 4)
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  else
    *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
}

// Operand hand-off to the next projection: x = hi + lo as two 16-bit values (the same split the
// projections' input preparation makes), hi in row r, lo in row mp + r of a [2][mp][ld] array.
template <typename W, int N>
__device__ __forceinline__ void store_hilo(void* xb, int r, int mp, int ld, size_t col, const float* v) {
  W* hi = reinterpret_cast<W*>(xb) + (size_t)r * ld + col;
  W* lo = reinterpret_cast<W*>(xb) + ((size_t)mp + r) * ld + col;
#pragma unroll
  for (int c = 0; c < N; ++c) {
    const W h = Io<W>::from_f(v[c]);
    hi[c] = h;
    lo[c] = Io<W>::from_f(v[c] - Io<W>::to_f(h));
  }
}

// Tiles [t0, t1) of split `split` out of n_tiles over ns splits.
__device__ __forceinline__ void split_tiles(int n_tiles, int split, int ns, int& t0, int& t1) {
  t0 = (int)((long long)n_tiles * split / ns);
  t1 = (int)((long long)n_tiles * (split + 1) / ns);
}

// The tile ring's reuse rule (see k_attention).  A CTA with ntile tiles, S slots and WQ query groups of
// kWarps / WQ warps: when no slot is refilled (ntile <= S) the ring uses all S slots and every warp set
// takes tiles; otherwise it uses R <= S slots (tile k in slot k % R) and WK warp sets with R % WK == 0, so
// that every tile of a slot goes to the warps that released the tile before it, the most warp sets that
// allows (then the most slots).
__host__ __device__ __forceinline__ void ring_plan(int ntile, int S, int WQ, int& R, int& WK) {
  const int wmax = kWarps / WQ;
  R = S;
  WK = wmax;
  if (ntile <= S) return;
  WK = 0;
  for (int r = S; r >= 1; --r) {
    int w = wmax < r ? wmax : r;
    while (r % w) --w;
    if (w > WK) {
      WK = w;
      R = r;
    }
  }
}

// QPW queries per warp: four (each key tile's K and V, read from shared memory once, serve four queries),
// or one for query blocks of at most four queries (one-row passes: GQA groups of four, MHA), where four
// warps then share the work of one group of four and no warp computes padding queries.
// Query groups of a CTA with nqc queries, QPW per warp: a power of two, so that kWarps / groups warps
// serve each group.
__host__ __device__ __forceinline__ int query_groups(int nqc, int qpw) {
  const int g = (nqc + qpw - 1) / qpw;
  return g <= 1 ? 1 : g <= 2 ? 2 : g <= 4 ? 4 : g <= 8 ? 8 : 16;
}
// Queries per warp of a launch whose query blocks hold at most nqc_max queries.
__host__ __device__ __forceinline__ int queries_per_warp(int nqc_max) { return nqc_max <= 4 ? 1 : 4; }

template <typename T, int HD, int QPW>
__global__ void __launch_bounds__(kWarps * 32, 1) k_attention(const __grid_constant__ CUtensorMap tk,
                                                              const __grid_constant__ CUtensorMap tv, AttnArgs a) {
  using G = TileGeo<T, HD>;
  constexpr int DPL = HD / 32;  // output dims per lane (lane owns dims lane*DPL ..)
  constexpr int PS = HD + 4;    // partial state: weighted V sum [HD], m, l, (pad): rows stay 16-byte aligned
  extern __shared__ unsigned char s_dyn[];
  __shared__ __align__(16) float s_q[kQB][HD];
  __shared__ __align__(16) float s_p[kWarps][kTile][QPW];  // softmax weights, QPW queries per key
  __shared__ __align__(8) uint64_t s_full[kMaxSlots];
  __shared__ int s_cons[kMaxSlots];
  __shared__ int s_fail;
  __shared__ unsigned s_shift;  // slots whose phases run one ahead: an early copy made under a stale hint
  // SWIZZLE_128B wants 1024-byte aligned boxes; the same offset in every CTA of the cluster
  unsigned char* ring = s_dyn + ((1024 - (smem_u32(s_dyn) & 1023)) & 1023);

  const int kvh = blockIdx.x, split = blockIdx.y, qblk = blockIdx.z, ns = gridDim.y;
  const int qb = a.qb;  // queries per query block (<= kQB)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.n_slots;
  const size_t layer_rows = (size_t)a.n_pages * a.n_kv * kPage;
  const T* kc = reinterpret_cast<const T*>(a.kcache) + (size_t)a.layer * layer_rows * HD;
  const T* vc = reinterpret_cast<const T*>(a.vcache) + (size_t)a.layer * layer_rows * HD;
  const int n_new = (a.rows + kTile - 1) / kTile;  // tiles of new slots (when they do not follow the prefix)
  // Key tiles of a pass whose prefix ends at p and whose new slots start at base: when base == p (every pass
  // but the DP's, whose rows sit at the target's position past the committed slots) the new slots continue
  // the prefix, and the keys [0, p + rows) are cut into tiles of 32 together; otherwise the prefix and the
  // new slots are tiled separately.  Every tile of the contiguous range comes in by TMA.
  auto n_tiles = [&](int p, bool contig) {
    return contig ? (p + a.rows + kTile - 1) / kTile : (p + kTile - 1) / kTile + n_new;
  };
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&s_full[i], 1);
      s_cons[i] = 0;
    }
    s_fail = 0;
    s_shift = 0;
    fence_barrier_init();
  }
  __syncthreads();

  griddep_launch();
  const int group = a.n_q / a.n_kv;
  const int nq = a.rows * group;
  const int nqc = min(qb, nq - qblk * qb);  // queries of this CTA
  const int WQ = query_groups(nqc, QPW);
  // Before the wait: the descriptor may still hold the previous pass's prefix (each pass rewrites it at
  // its start), so what is done here under that hint is checked after the wait.  An L2 prefetch only
  // warms the cache: this CTA's prefix tiles, found through the block table (never written on the
  // device).  With a.early warp s also fills ring slot s (TMA) with the CTA's s-th tile when that is a
  // prefix tile whose keys all lie below the committed length: no kernel that may still be running
  // writes them.  A copy made under a stale hint is let land and its slot refilled.  (None of it when a
  // draft exit has already closed this forward's gate.)
  const bool warm = gate_open(a.gate);
  auto tma_tile = [&](int slot, int row) {  // one lane: the 32 key rows from cache row `row` into `slot`
    unsigned char* sl = ring + (size_t)slot * G::kSlot;
    mbar_expect_tx(&s_full[slot], (uint32_t)G::kSlot);
#pragma unroll
    for (int bx = 0; bx < G::kBoxes; ++bx) {
      tma_load_rows(sl + bx * kBoxBytes, &tk, bx * (128 / (int)sizeof(T)), row, &s_full[slot]);
      tma_load_rows(sl + G::kHalf + bx * kBoxBytes, &tv, bx * (128 / (int)sizeof(T)), row, &s_full[slot]);
    }
  };
  // Warps may read different hints (the descriptor can change meanwhile): each decides for its own slot.
  int row_hint = -1;  // cache row of the tile slot `warp` takes first, under the hint
  bool early;         // slot `warp` was filled before the wait
  const int hint = min(*reinterpret_cast<const volatile int*>(&a.desc->prefix), a.n_pages * kPage);
  const bool contig_h = *reinterpret_cast<const volatile int*>(&a.desc->base) == hint;
  {
    const int tc = a.early && warm ? *reinterpret_cast<const volatile int*>(a.committed) : 0;
    const int hint_pt = contig_h ? n_tiles(hint, true) : (hint + kTile - 1) / kTile;  // tiles loaded by TMA
    int hb, he, Rh, WKh;
    split_tiles(n_tiles(hint, contig_h), split, ns, hb, he);
    ring_plan(he - hb, S, WQ, Rh, WKh);
    int n_early = 0;  // tiles hb .. hb + n_early - 1 go to slots 0 .. n_early - 1 before the wait
    if (a.early && warm) {
      // tiles [0, last) use keys below tc only (a contiguous range's tile that reaches the new slots does not)
      const int last = contig_h ? min(tc, hint) / kTile : tc >= hint ? hint_pt : tc / kTile;
      n_early = max(0, min(min(last, he), hb + Rh) - hb);
    }
    if (lane == 0 && warp < S && hb + warp < min(he, hint_pt)) {
      const int key = (hb + warp) * kTile;
      row_hint = (a.btab[key / kPage] * a.n_kv + kvh) * kPage + (key % kPage);
    }
    early = warp < n_early;
    if (early && lane == 0) tma_tile(warp, row_hint);
    if (warm) {
      const int hp = min(he, hint_pt);
      for (int i = threadIdx.x; i < 2 * (hp - hb - n_early); i += blockDim.x) {
        const int ti = hb + n_early + (i >> 1), key = ti * kTile;
        const size_t row = ((size_t)a.btab[key / kPage] * a.n_kv + kvh) * kPage + (key % kPage);
        l2_prefetch(((i & 1) ? vc : kc) + row * HD, (uint32_t)(kTile * G::kRowBytes));
      }
      l2_prefetch_share(a.pf, a.pf_bytes, (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x,
                        gridDim.x * gridDim.y * gridDim.z);
    }
  }
  trace_mark(a.trace, 0);
  griddep_wait();
  if (!gate_open(a.gate)) {  // every CTA of the cluster reads the same word: all return together
    if (early && !mbar_wait_bounded(&s_full[warp], 0u) && lane == 0 && a.err) atomicExch(a.err, 1);
    return;  // (a copy issued before the wait has landed first)
  }
  trace_mark(a.trace, 1);

  // queries of this CTA (written by the projection just before): index qi = r * group + g -> row r, head
  // kvh*group + g.  Loaded into registers first, so their latency overlaps the descriptor read below.
  constexpr int QV = kQB * HD / 4 / (kWarps * 32);  // float4 per thread
  float4 qreg[QV];
#pragma unroll
  for (int it = 0; it < QV; ++it) {
    const int i = (it * kWarps * 32 + threadIdx.x) * 4;
    const int ql = i / HD, dd = i - ql * HD;
    const int qi = qblk * qb + ql;
    qreg[it] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (ql < qb && qi < nq) {
      const int r = qi / group, h = kvh * group + (qi - r * group);
      qreg[it] = *reinterpret_cast<const float4*>(a.q + (size_t)r * a.n_q * HD + h * HD + dd);
    }
  }

  const PassDesc* d = a.desc;
  const int prefix = d->prefix, base = d->base;
  const bool contig = base == prefix;
  const int pt = contig ? n_tiles(prefix, true) : (prefix + kTile - 1) / kTile;  // tiles loaded by TMA
  int tb, te;
  split_tiles(n_tiles(prefix, contig), split, ns, tb, te);

  // Load tile ti into ring slot `slot` (one warp): prefix tiles (and every tile of a contiguous range) by
  // TMA, separately tiled new slots (just written by the QKV projection, anywhere in their pages) by
  // cp.async.  Either way one phase of s_full[slot] completes when it lands.
  auto fill = [&](int slot, int ti, int row) {
    unsigned char* sl = ring + (size_t)slot * G::kSlot;
    if (ti < pt) {
      if (lane == 0) {
        if (row < 0) {
          const int key = ti * kTile;
          row = (a.btab[key / kPage] * a.n_kv + kvh) * kPage + (key % kPage);
        }
        tma_tile(slot, row);
      }
    } else {
      const int e0 = (ti - pt) * kTile;
      for (int idx = lane; idx < kTile * G::kChunks; idx += 32) {
        const int r = idx / G::kChunks, c = idx - r * G::kChunks;
        const int e = e0 + r;
        if (e < a.rows) {  // rows past the last new slot stay stale: never read as values, scores masked
          const size_t gi = kv_index(a.layer, base + e, kvh, c * G::kChunk, a.btab, a.n_pages, a.n_kv, HD);
          cp_async16(sl + swz(r, c * 16), reinterpret_cast<const T*>(a.kcache) + gi);
          cp_async16(sl + G::kHalf + swz(r, c * 16), reinterpret_cast<const T*>(a.vcache) + gi);
        }
      }
      cp_async_arrive(&s_full[slot]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_full[slot]);
    }
  };
  // A slot holds this CTA's tiles k, k + R, k + 2R, ... (R slots in use).  A parity wait only tells
  // consecutive phases of a slot apart, so when slots are reused every tile of a slot must go to the
  // same warps, the ones that released the tile before it: the tiles are shared among WK warp sets with
  // R % WK == 0 (ring_plan).  Warp roles: query group wq (QPW queries) of WQ, tile share wk of WK.
  int R, WK;
  ring_plan(te - tb, S, WQ, R, WK);
  // A slot filled before the wait under this warp's hint, when that was the prefix (and the same tiling),
  // holds tile tb + warp already (same split, same ring plan); under a stale hint its copy lands first and
  // the slot's next phase brings the real tile.
  const bool stale = prefix != hint || contig != contig_h;
  if (early && stale) {
    if (!mbar_wait_bounded(&s_full[warp], 0u) && lane == 0 && a.err) atomicExch(a.err, 1);
    fence_proxy_async();
    if (lane == 0) atomicOr(&s_shift, 1u << warp);
  }
  if (warp < R && tb + warp < te && !(early && !stale))
    fill(warp, tb + warp, !stale ? __shfl_sync(0xffffffffu, row_hint, 0) : -1);

  if (a.head_pf) {  // the heads of the next matrix's rows into L2, one prefetch per thread at most
    const int cid = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    const int nt = gridDim.x * gridDim.y * gridDim.z * blockDim.x;
    for (int r = cid * blockDim.x + threadIdx.x; r < a.head_rows; r += nt)
      l2_prefetch(a.head_pf + (size_t)r * a.head_stride, (uint32_t)a.head_bytes);
  }
  const float scale = rsqrtf((float)HD);
#pragma unroll
  for (int it = 0; it < QV; ++it) {
    const int i = (it * kWarps * 32 + threadIdx.x) * 4;
    const int ql = i / HD, dd = i - ql * HD;
    float4 v = qreg[it];
    v.x *= scale;
    v.y *= scale;
    v.z *= scale;
    v.w *= scale;
    *reinterpret_cast<float4*>(&s_q[ql][dd]) = v;
  }
  __syncthreads();

  const unsigned shifted = s_shift;
  const int wq = warp % WQ, wk = warp / WQ;  // warps with wk >= WK take no tile
  float m_run[QPW], l_run[QPW], acc[QPW][DPL];
  bool qvalid[QPW];
  unsigned long long qmask[QPW];
#pragma unroll
  for (int j = 0; j < QPW; ++j) {
    m_run[j] = -INFINITY;
    l_run[j] = 0.f;
#pragma unroll
    for (int c = 0; c < DPL; ++c) acc[j][c] = 0.f;
    const int qi = qblk * qb + wq * QPW + j;
    qvalid[j] = wq * QPW + j < nqc;
    qmask[j] = qvalid[j] ? d->mask[qi / group] : 0ull;
  }
  const float* sq = &s_q[wq * QPW][0];

  for (int ti = wk < WK ? tb + wk : te; ti < te; ti += WK) {
    const int k = ti - tb, slot = k % R;
    if (*reinterpret_cast<volatile int*>(&s_fail)) break;
    const uint32_t par = (uint32_t)(k / R + ((shifted >> slot) & 1u)) & 1u;
    if (!mbar_wait_bounded(&s_full[slot], par)) {
      if (lane == 0) {
        s_fail = 1;
        if (a.err) atomicExch(a.err, 1);
      }
      mbar_wait_bounded(&s_full[slot], par);  // one more bounded wait for the copy in flight
      break;
    }
    // keys of the tile: nvalid of them; key lane is new slot e0 + lane when that is >= 0, else a prefix key
    int nvalid, e0;
    if (contig) {
      nvalid = min(kTile, prefix + a.rows - ti * kTile);
      e0 = ti * kTile - prefix;
    } else if (ti < pt) {
      nvalid = min(kTile, prefix - ti * kTile);
      e0 = -kTile;
    } else {
      nvalid = min(kTile, a.rows - (ti - pt) * kTile);
      e0 = (ti - pt) * kTile;
    }
    const unsigned char* kt = ring + (size_t)slot * G::kSlot;
    const unsigned char* vt = kt + G::kHalf;

    // scores: lane = key of the tile; four partial sums per query keep the FMA chains short
    float dot[QPW][4];
#pragma unroll
    for (int j = 0; j < QPW; ++j) dot[j][0] = dot[j][1] = dot[j][2] = dot[j][3] = 0.f;
#pragma unroll 4
    for (int c = 0; c < G::kChunks; ++c) {
      const uint4 raw = *reinterpret_cast<const uint4*>(kt + swz(lane, c * 16));
      float kf[G::kChunk];
      unpack16<T>(raw, kf);
#pragma unroll
      for (int h = 0; h < G::kChunk; h += 4) {
#pragma unroll
        for (int j = 0; j < QPW; ++j) {
          const float4 qv = *reinterpret_cast<const float4*>(sq + j * HD + c * G::kChunk + h);
          dot[j][0] = fmaf(qv.x, kf[h], dot[j][0]);
          dot[j][1] = fmaf(qv.y, kf[h + 1], dot[j][1]);
          dot[j][2] = fmaf(qv.z, kf[h + 2], dot[j][2]);
          dot[j][3] = fmaf(qv.w, kf[h + 3], dot[j][3]);
        }
      }
    }
    // online softmax update of the warp's queries, their warp reductions interleaved
    float sc[QPW], mx[QPW];
#pragma unroll
    for (int j = 0; j < QPW; ++j) {
      const bool vis = qvalid[j] && lane < nvalid && (e0 + lane < 0 || ((qmask[j] >> (e0 + lane)) & 1ull));
      sc[j] = vis ? (dot[j][0] + dot[j][1]) + (dot[j][2] + dot[j][3]) : -INFINITY;
      mx[j] = sc[j];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
      for (int j = 0; j < QPW; ++j) mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], o));
    }
    float p[QPW], corr[QPW], ps[QPW];
#pragma unroll
    for (int j = 0; j < QPW; ++j) {
      const float m_new = fmaxf(m_run[j], mx[j]);
      // no visible key yet: nothing to rescale (and exp(-inf - -inf) would be NaN)
      corr[j] = m_new == -INFINITY ? 1.f : expf(m_run[j] - m_new);
      p[j] = sc[j] == -INFINITY ? 0.f : expf(sc[j] - m_new);
      ps[j] = p[j];
      m_run[j] = m_new;
    }
    if constexpr (QPW == 4)
      *reinterpret_cast<float4*>(&s_p[warp][lane][0]) = make_float4(p[0], p[1], p[2], p[3]);
    else
      s_p[warp][lane][0] = p[0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
      for (int j = 0; j < QPW; ++j) ps[j] += __shfl_xor_sync(0xffffffffu, ps[j], o);
    }
#pragma unroll
    for (int j = 0; j < QPW; ++j) {
      l_run[j] = fmaf(l_run[j], corr[j], ps[j]);
#pragma unroll
      for (int c = 0; c < DPL; ++c) acc[j][c] *= corr[j];
    }
    __syncwarp();
    // weighted V sum: lane = dims lane*DPL ..; rows past nvalid are never read
    const int xb = lane * DPL * (int)sizeof(T);
#pragma unroll 4
    for (int kk = 0; kk < nvalid; ++kk) {
      float v[DPL];
      lds_elems<T, DPL>(vt + swz(kk, xb), v);
      float pj[QPW];
      if constexpr (QPW == 4) {
        const float4 pk = *reinterpret_cast<const float4*>(&s_p[warp][kk][0]);
        pj[0] = pk.x, pj[1] = pk.y, pj[2] = pk.z, pj[3] = pk.w;
      } else {
        pj[0] = s_p[warp][kk][0];
      }
#pragma unroll
      for (int j = 0; j < QPW; ++j) {
#pragma unroll
        for (int c = 0; c < DPL; ++c) acc[j][c] = fmaf(pj[j], v[c], acc[j][c]);
      }
    }
    __syncwarp();
    // release the slot; its last consumer refills it with tile ti + R
    int last = 0;
    if (lane == 0) {
      __threadfence_block();
      last = atomicAdd(&s_cons[slot], 1) == WQ - 1;
      if (last) {
        s_cons[slot] = 0;
        __threadfence_block();
      }
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last && ti + R < te) {
      fence_proxy_async();  // the consumers' reads of the slot come before the copies that overwrite it
      fill(slot, ti + R, -1);
    }
  }
  __syncthreads();  // the ring is free: it now holds the partial states

  // Partial states: per warp [warp][j], then per CTA query [ql] (the WK
  // warps of a query group combined in a fixed order), then the cluster
  // merge over distributed shared memory, queries spread over the ranks.
  float* s_wpart = reinterpret_cast<float*>(ring);    // [kWarps * QPW][PS]
  float* s_cpart = s_wpart + kWarps * 4 * PS;          // [kQB][PS]
#pragma unroll
  for (int j = 0; j < QPW; ++j) {
    float* pp = s_wpart + (warp * QPW + j) * PS;
    if (lane == 0) {
      pp[HD] = m_run[j];
      pp[HD + 1] = l_run[j];
    }
    store_dims<DPL>(pp + lane * DPL, acc[j]);
  }
  __syncthreads();
  for (int ql = warp; ql < nqc; ql += kWarps) {
    const int qg = ql / QPW, j = ql % QPW;
    float M = -INFINITY;
    for (int w = 0; w < WK; ++w) M = fmaxf(M, s_wpart[((qg + WQ * w) * QPW + j) * PS + HD]);
    float L = 0.f, o[DPL];
#pragma unroll
    for (int c = 0; c < DPL; ++c) o[c] = 0.f;
    for (int w = 0; w < WK; ++w) {
      const float* pp = s_wpart + ((qg + WQ * w) * QPW + j) * PS;
      const float wt = pp[HD] == -INFINITY ? 0.f : expf(pp[HD] - M);
      L = fmaf(pp[HD + 1], wt, L);
      float v[DPL];
      load_dims<DPL>(pp + lane * DPL, v);
#pragma unroll
      for (int c = 0; c < DPL; ++c) o[c] = fmaf(wt, v[c], o[c]);
    }
    float* cp = s_cpart + ql * PS;
    if (lane == 0) {
      cp[HD] = M;
      cp[HD + 1] = L;
    }
    store_dims<DPL>(cp + lane * DPL, o);
  }

  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  const int nsp = (int)cluster.num_blocks(), rank = (int)cluster.block_rank();
  for (int ql = rank + nsp * warp; ql < nqc; ql += nsp * kWarps) {
    const int qi = qblk * qb + ql;
    float ms = -INFINITY, lsum = 0.f;
    if (lane < nsp) {
      const float* rp = cluster.map_shared_rank(s_cpart + ql * PS, (unsigned)lane);
      ms = rp[HD];
      lsum = rp[HD + 1];
    }
    float vals[8][DPL];
#pragma unroll
    for (int sp = 0; sp < 8; ++sp) {
      if (sp < nsp) load_dims<DPL>(cluster.map_shared_rank(s_cpart + ql * PS, (unsigned)sp) + lane * DPL, vals[sp]);
    }
    const float M = warp_max(ms);
    const float w = (ms == -INFINITY) ? 0.f : expf(ms - M);
    const float L = warp_sum(lsum * w);
    float o[DPL];
#pragma unroll
    for (int c = 0; c < DPL; ++c) o[c] = 0.f;
#pragma unroll
    for (int sp = 0; sp < 8; ++sp) {
      if (sp < nsp) {
        const float ws = __shfl_sync(0xffffffffu, w, sp);
#pragma unroll
        for (int c = 0; c < DPL; ++c) o[c] = fmaf(ws, vals[sp][c], o[c]);
      }
    }
    const int r = qi / group, h = kvh * group + (qi - r * group);
    const float invL = L > 0.f ? 1.0f / L : 0.f;
#pragma unroll
    for (int c = 0; c < DPL; ++c) o[c] *= invL;
    const size_t col = (size_t)h * HD + lane * DPL;
    store_dims<DPL>(a.out + (size_t)r * a.n_q * HD + col, o);
    if (a.xb_next) {
      if (a.xb_fp16)
        store_hilo<__half, DPL>(a.xb_next, r, a.next_mp, a.n_q * HD, col, o);
      else
        store_hilo<__nv_bfloat16, DPL>(a.xb_next, r, a.next_mp, a.n_q * HD, col, o);
    }
  }
  cluster.sync();  // every CTA's shared memory stays alive until all ranks have read it
  trace_mark(a.trace, 2);
}

namespace {

int device_sms() {
  static int sms = 0;
  if (!sms) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) ==
                                                   cudaSuccess && n > 0)
      sms = n;
    else
      return 148;
  }
  return sms;
}

}  // namespace


namespace {

template <typename T, int HD>
constexpr size_t attn_smem(int slots) {
  using G = TileGeo<T, HD>;
  return 1024 + std::max((size_t)slots * G::kSlot, (size_t)G::kPartBytes);
}

template <typename T, int HD>
bool set_attn_attr() {
  const int bytes = (int)attn_smem<T, HD>(TileGeo<T, HD>::kSlots);
  return cudaFuncSetAttribute(k_attention<T, HD, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) ==
             cudaSuccess &&
         cudaFuncSetAttribute(k_attention<T, HD, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) ==
             cudaSuccess;
}

// Clusters of each size (1, 2, 4, 8 CTAs) that can be resident at once, per element type, head size and
// ring slots (shared memory), from the occupancy calculator; 0 = unknown.
int g_max_clusters[3][2][4][kMaxSlots + 1];

template <typename T, int HD>
void fill_max_clusters(int ti, int hi) {
  for (int li = 0; li < 4; ++li)
    for (int slots = 1; slots <= TileGeo<T, HD>::kSlots; ++slots) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 1;
      attr[0].val.clusterDim.y = 1u << li;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(1, 1u << li, 1);
      cfg.blockDim = dim3(kWarps * 32);
      cfg.dynamicSmemBytes = attn_smem<T, HD>(slots);
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, k_attention<T, HD, 4>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
      }
      g_max_clusters[ti][hi][li][slots] = n;
    }
}

bool attn_attrs() {
  static std::once_flag once;
  static bool ok = false;
  std::call_once(once, [] {
    ok = set_attn_attr<float, 64>() && set_attn_attr<float, 128>() && set_attn_attr<__half, 64>() &&
         set_attn_attr<__half, 128>() && set_attn_attr<__nv_bfloat16, 64>() && set_attn_attr<__nv_bfloat16, 128>();
    if (ok) {
      fill_max_clusters<__nv_bfloat16, 64>(0, 0);
      fill_max_clusters<__nv_bfloat16, 128>(0, 1);
      fill_max_clusters<__half, 64>(1, 0);
      fill_max_clusters<__half, 128>(1, 1);
      fill_max_clusters<float, 64>(2, 0);
      fill_max_clusters<float, 128>(2, 1);
    }
  });
  return ok;
}

// Ring slots of a launch: the shared-memory budget's, or fewer under a ring cap (bytes, 0 = none).
int ring_slots_of(int kv_type, int hd, int ring_cap) {
  const int slots = kv_type == 2 ? (hd == 128 ? TileGeo<float, 128>::kSlots : TileGeo<float, 64>::kSlots)
                                 : (hd == 128 ? TileGeo<__half, 128>::kSlots : TileGeo<__half, 64>::kSlots);
  const int slot_bytes = kv_type == 2 ? (hd == 128 ? TileGeo<float, 128>::kSlot : TileGeo<float, 64>::kSlot)
                                      : (hd == 128 ? TileGeo<__half, 128>::kSlot : TileGeo<__half, 64>::kSlot);
  return ring_cap > 0 ? std::max(1, std::min(slots, ring_cap / slot_bytes)) : slots;
}

}  // namespace

void attention_layout(int max_keys, int rows, int group, int n_kv, int kv_type, int hd, int ring_cap, int* qb_out,
                      int* ns_out) {
  // Every (query block size, key splits) pair is scored per wave of clusters (the occupancy
  // calculator's count of clusters of that size and ring that fit at once) by a two-term time model:
  // the CTA's query x key-tile products (the SM's issue load) plus the tiles one warp handles in
  // sequence (each warp scores four queries per tile; the warps sharing a query group split the tiles,
  // at most R of them when the ring's R slots are refilled), weighted 1 : 19 as fitted to timings of
  // four layouts of a 7-row verify over 900 keys on GB300 (0.105 us per query-tile, 2.0 us per tile in
  // sequence), plus 40 per wave (about 4 us of start-up and cluster merge that every wave pays: fitted to
  // one-row launches of the 13B shape, 40 KV heads, where one wave of 2-CTA clusters took 10.3 us and
  // three waves of 8-CTA clusters 23.2 us).  Ties go to fewer CTAs (fewer copies of each key tile), then
  // the larger query block.
  attn_attrs();
  const int tiles = (max_keys + kTile - 1) / kTile + 1;
  const int sms = device_sms();
  const int nq = rows * group;
  const int ti = kv_type == 2 ? 2 : kv_type == 1 ? 1 : 0, hi = hd == 128 ? 1 : 0;
  const int kslots = ring_slots_of(kv_type, hd, ring_cap);
  long long best = -1, best_ctas = 0;
  for (int qb = kQB; qb >= 4; qb /= 2) {
    const int qblocks = (nq + qb - 1) / qb;
    const int nqc = std::min(qb, nq);
    const int wq_groups = query_groups(nqc, queries_per_warp(nqc));  // query groups per CTA
    for (int li = 0; li < 4; ++li) {
      const int ns = 1 << li;
      if (ns > 1 && 2 * ns > tiles) break;
      const int tc = (tiles + ns - 1) / ns;  // tiles per CTA
      const int slots = std::max(1, std::min(kslots, tc));
      const long long clusters = (long long)n_kv * qblocks;
      int maxc = g_max_clusters[ti][hi][li][slots];
      if (maxc < 1) maxc = std::max(1, sms / ns);
      const long long waves = (clusters + maxc - 1) / maxc;
      int r, wk_eff;
      ring_plan(tc, slots, wq_groups, r, wk_eff);
      const long long per_warp = (tc + wk_eff - 1) / wk_eff;
      const long long work = waves * ((long long)nqc * tc + 19 * per_warp + 40), ctas = clusters * ns;
      if (best < 0 || work < best || (work == best && ctas < best_ctas)) {
        best = work;
        best_ctas = ctas;
        *qb_out = qb;
        *ns_out = ns;
      }
    }
  }
}

namespace {

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
  if (a.ring_cap > 0) a.n_slots = std::max(1, std::min(a.n_slots, a.ring_cap / G::kSlot));
  const int group = a.n_q / a.n_kv;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;  // the splits of one (kv head, query block)
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = a.n_split;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(a.n_kv, a.n_split, (a.rows * group + a.qb - 1) / a.qb);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = attn_smem<T, HD>(a.n_slots);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = g_pdl ? 2 : 1;
  g_launches += 1;
  if (queries_per_warp(std::min(a.qb, a.rows * group)) == 1)
    return cudaLaunchKernelEx(&cfg, k_attention<T, HD, 1>, tk, tv, a) == cudaSuccess;
  return cudaLaunchKernelEx(&cfg, k_attention<T, HD, 4>, tk, tv, a) == cudaSuccess;
}

template <typename T>
bool run_attn_hd(const AttnArgs& a, cudaStream_t st) {
  return a.hd == 128 ? run_attn<T, 128>(a, st) : run_attn<T, 64>(a, st);
}

}  // namespace

bool init_attention_kernels() { return attn_attrs(); }

namespace {
// The standalone attention's row descriptor, passed by value and stored into the caller's device scratch.
__global__ void k_store_desc(const __grid_constant__ PassDesc d, PassDesc* out) {
  const unsigned* src = reinterpret_cast<const unsigned*>(&d);
  unsigned* dst = reinterpret_cast<unsigned*>(out);
  for (int i = threadIdx.x; i < (int)(sizeof(PassDesc) / 4); i += blockDim.x) dst[i] = src[i];
}
}  // namespace

bool launch_store_desc(const PassDesc& d, PassDesc* out, cudaStream_t st) {
  static_assert(sizeof(PassDesc) % 4 == 0, "the descriptor is copied as 32-bit words");
  g_launches += 1;
  k_store_desc<<<1, 128, 0, st>>>(d, out);
  return cudaGetLastError() == cudaSuccess;
}

bool launch_attention(const AttnArgs& a, int kv_type, cudaStream_t st) {
  if (a.n_split < 1 || a.n_split > 8 || a.rows < 1 || a.rows > kMaxRows || (a.hd != 64 && a.hd != 128) ||
      a.qb < 1 || a.qb > kQB)
    return false;
  if (((uintptr_t)a.kcache | (uintptr_t)a.vcache) & 15) return false;  // TMA wants 16-byte aligned tensors
  if (kv_type == 2) return run_attn_hd<float>(a, st);
  if (kv_type == 1) return run_attn_hd<__half>(a, st);
  return run_attn_hd<__nv_bfloat16>(a, st);
}

}  // namespace ssd

extern "C" void ssd_attn_ring_rule(int ntile, int S, int WQ, int* R, int* WK) {
  if (ntile < 0 || S < 1 || WQ < 1 || WQ > ssd::kWarps) return;
  int r, w;
  ssd::ring_plan(ntile, S, WQ, r, w);
  if (R) *R = r;
  if (WK) *WK = w;
}
