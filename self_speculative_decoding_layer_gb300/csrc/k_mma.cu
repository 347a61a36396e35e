// Tensor-core (tcgen05) projections for 2..64 input rows: the verify pass
// (K+1 rows), tree verification (N+1 rows), the CLaSp DP rows and prefill
// chunks.
//
// Y[M, N] = X[M, K] W[N, K]^T is computed as D[128, 2 Mpad] = W_tile [X_hi; X_lo]^T
// ("swap AB"): 128 weight rows fill the MMA's M dimension and the few input
// rows are its N dimension (Mpad = M rounded up to 8, 16, 32, 48 or 64).  The
// input rows are first prepared by k_act_prep (or handed over by the kernel
// that produced them) -- the same RMSNorm / int8 arithmetic as the CUDA-core
// kernels -- and stored as 16-bit operands: a hi/lo pair (x = hi + lo, both
// bf16 or both fp16 like the weights), multiplied by one MMA of width 2 Mpad,
// which keeps the activation at close to fp32 precision; or the int8 codes
// (exact in 16 bits, width Mpad, so Mpad >= 16) with a per-row scale.
//
// Two work distributions.  Split-K in a cluster (k_mma_split, used when the
// matrix has at most one output tile per SM): one output tile per
// thread-block cluster of C CTAs, rank r streaming its C-th of the K stages
// into its own TMEM accumulator; the ranks then add their partial tiles over
// distributed shared memory (each rank the same share of the tile's output
// units, summing the C partials in rank order) and run the epilogue of those
// units, so no partial tile goes through L2 and no CTA merges alone.
// Stream-K (k_mma, matrices with more tiles than SMs: the lm_head and the
// widest projections): the (weight tile, 64-wide K stage) items of the whole
// matrix are cut into one equal contiguous run per CTA, one CTA per SM, so
// every SM streams the same number of weight bytes whatever the matrix shape.  A run
// covers parts of one or more tiles ("segments").  A producer warp keeps a
// deep TMA (SWIZZLE_128B) + mbarrier ring full, one thread issues
// tcgen05.mma into one of two TMEM accumulators (the epilogue of a segment
// overlaps the MMAs of the next), and four epilogue warps drain TMEM.  A tile
// cut between CTAs is summed by the CTA that completes it, in CTA order; the
// epilogue is the one of the CUDA-core kernels (RoPE + KV write, residual,
// SwiGLU, logits).
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>
#include <type_traits>

#include "../../include/ssd.h"
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace ssd {

bool init_linear_kernels();

constexpr int kBK = 64;             // K elements per stage (one 128-byte swizzle row)
constexpr int kWT = 128 * kBK * 2;  // bytes of one 128-row weight tile stage

// ---------------------------------------------------------------- input preparation

struct PrepArgs {
  const float* X;
  int ldx, M, Mpad, K;
  const void* gamma;
  float eps;
  int int8;
  void* xb;      // [2][Mpad][K] 16-bit: hi rows, then lo rows
  float* scale;  // [Mpad]: int8 scale per row (1 otherwise)
  unsigned long long* trace;
};

__device__ __forceinline__ float block_sum_or_max(float v, float* red, bool is_max) {
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
__global__ void __launch_bounds__(256) k_act_prep(PrepArgs a) {
  __shared__ float red[32];
  griddep_launch();
  trace_mark(a.trace, 0);
  griddep_wait();
  trace_mark(a.trace, 1);
  const int m = blockIdx.x;
  T* hi = reinterpret_cast<T*>(a.xb) + (size_t)m * a.K;
  T* lo = reinterpret_cast<T*>(a.xb) + ((size_t)a.Mpad + m) * a.K;
  if (m >= a.M) {  // padding rows are zero
    for (int k = threadIdx.x; k < a.K; k += blockDim.x) {
      hi[k] = Io<T>::from_f(0.f);
      lo[k] = Io<T>::from_f(0.f);
    }
    if (threadIdx.x == 0) a.scale[m] = 0.f;
    trace_mark(a.trace, 2);
    return;
  }
  const float* x = a.X + (size_t)m * a.ldx;
  const T* g = reinterpret_cast<const T*>(a.gamma);
  float inv = 1.f;
  if (g) {
    float ss = 0.f;
    for (int k = threadIdx.x * 8; k < a.K; k += blockDim.x * 8) {
      const float4* xp = reinterpret_cast<const float4*>(x + k);
      const float4 u = xp[0], v = xp[1];
      ss += u.x * u.x + u.y * u.y + u.z * u.z + u.w * u.w + v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    ss = block_sum_or_max(ss, red, false);
    inv = 1.0f / sqrtf(ss / (float)a.K + a.eps);
  }
  float qm = 0.f, qs = 1.f;
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
    amax = block_sum_or_max(amax, red, true);
    qs = 0.f;
    if (amax > 0.f) {
      qm = __fdiv_rn(127.0f, amax);
      qs = __fdiv_rn(amax, 127.0f);
    }
  }
  for (int k = threadIdx.x * 8; k < a.K; k += blockDim.x * 8) {
    const float4* xp = reinterpret_cast<const float4*>(x + k);
    const float4 u = xp[0], v = xp[1];
    float xv[8] = {u.x, u.y, u.z, u.w, v.x, v.y, v.z, v.w};
    float gv[8];
    if (g) Io<T>::unpack8(*reinterpret_cast<const uint4*>(g + k), gv);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float z = g ? xv[e] * inv * gv[e] : xv[e];
      if (a.int8) z = q8_code(z, qm);
      const T h = Io<T>::from_f(z);
      hi[k + e] = h;
      lo[k + e] = a.int8 ? Io<T>::from_f(0.f) : Io<T>::from_f(z - Io<T>::to_f(h));
    }
  }
  if (threadIdx.x == 0) a.scale[m] = a.int8 ? qs : 1.f;
  trace_mark(a.trace, 2);
}

// ---------------------------------------------------------------- tcgen05 helpers

// Shared-memory matrix descriptor of a K-major tile with 128-byte rows in the
// 128-byte swizzle (8-row atoms of 1024 bytes, tile base 1024-byte aligned).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | (1ull << 16) | (64ull << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator, A and B of one 16-bit
// type (bf16 or fp16), both K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc_f16(int n, bool bf16) {
  const uint32_t fmt = bf16 ? 1u : 0u;
  return (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
          tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_cta(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Columns of the accumulators: one MMA of N = 2 * Mpad multiplies a weight tile by the hi rows and the lo rows
// together (they are adjacent in shared memory), so a unit's accumulator holds W.hi in its first Mpad columns
// and W.lo in the next Mpad; int8 rows (no lo part) use the first Mpad only.
__host__ __device__ constexpr uint32_t tmem_pow2(uint32_t cols) {
  return cols <= 32 ? 32 : cols <= 64 ? 64 : cols <= 128 ? 128 : cols <= 256 ? 256 : 512;
}

// 16 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* out) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) out[i] = __uint_as_float(r[i]);
}

// out = columns [a, a+8) + columns [b, b+8) (the hi and lo halves of an 8-row accumulator), one wait for both.
__device__ __forceinline__ void tmem_ld8_sum(uint32_t ta, uint32_t tb, float* out) {
  uint32_t r[8], q[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(ta));
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3]), "=r"(q[4]), "=r"(q[5]), "=r"(q[6]), "=r"(q[7])
               : "r"(tb));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) out[i] = __uint_as_float(r[i]) + __uint_as_float(q[i]);
}

// out = columns [a, a+16) + columns [b, b+16) (the hi and lo halves of an accumulator), one wait for both.
__device__ __forceinline__ void tmem_ld16_sum(uint32_t ta, uint32_t tb, float* out) {
  uint32_t r[16], q[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(ta));
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3]), "=r"(q[4]), "=r"(q[5]), "=r"(q[6]), "=r"(q[7]), "=r"(q[8]),
        "=r"(q[9]), "=r"(q[10]), "=r"(q[11]), "=r"(q[12]), "=r"(q[13]), "=r"(q[14]), "=r"(q[15])
      : "r"(tb));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) out[i] = __uint_as_float(r[i]) + __uint_as_float(q[i]);
}

// ---------------------------------------------------------------- the GEMM kernel

struct MmaArgs {
  int M, K;
  int n_tiles;  // 128-row weight tiles (SwiGLU: gate/up tile pairs)
  int stages;   // K stages of kBK elements per tile
  int int8;
  const float* scale;
  float* part;    // partial tiles [CTA][first/last segment][NT][Mpad][128]
  int* counters;  // [n_tiles], zero between launches
  LinearArgs ep;  // epilogue targets
};

constexpr int kMmaSmemBudget = 216 * 1024;

// Operand rows read per TMEM load in the epilogue: 16 columns, or 8 for 8-row operands (an MMA of 128 rows
// needs N = 2 * MP to be a multiple of 16, so 8-row operands are always hi/lo pairs, never int8 codes).
template <int MP>
constexpr int acc_chunk() { return MP >= 16 ? 16 : 8; }

// Columns [c, c + acc_chunk) of one accumulator unit (TMEM address col) as fp32 rows: int8 codes as they
// are, hi/lo operands as the sum of the hi half and the lo half MP columns further on.
template <int MP>
__device__ __forceinline__ void tmem_acc(uint32_t col, bool int8, float* out) {
  if constexpr (MP >= 16) {
    if (int8)
      tmem_ld16(col, out);
    else
      tmem_ld16_sum(col, col + MP, out);
  } else {
    tmem_ld8_sum(col, col + MP, out);
  }
}

template <int MP, int NT>
struct MmaSmem {
  static constexpr int XT = MP * kBK * 2;                // one activation operand tile (hi or lo)
  static constexpr int kStage = NT * kWT + 2 * XT;      // one ring stage
  static constexpr int kC = NT * MP * 128 * 4;           // epilogue staging of one tile
  static constexpr int kE = NT == 1 ? MP * 128 * 4 + MP * 16 + 128 * 4 : MP * 16;  // epilogue inputs (see k_mma)
  static constexpr int kS0 = (kMmaSmemBudget - 2048 - kC - kE) / kStage;
  static constexpr int kStages = kS0 > 8 ? 8 : kS0;      // ring depth
  static constexpr int kBars = (2 * kStages + 4) * 8 + 16;
  static constexpr int kBytes = 1024 + kStages * kStage + kC + kE + kBars;
};

// epi_apply for the residual and QKV epilogues with their global inputs (residual rows, RoPE cos/sin,
// cache page) already staged in shared memory by the epilogue warps while the tile's MMAs ran.
template <typename T, int MP>
__device__ __forceinline__ void epi_staged(const LinearArgs& a, int m, int u, float y0, float y1, int n0, float* E,
                                           const int* e_page, const int* e_sidx, const float* e_gamma) {
  if (a.epi == EPI_RESID) {
    const int lr = 2 * u - n0;
    const float h0 = E[m * 128 + lr] + y0, h1 = E[m * 128 + lr + 1] + y1;
    float* h = a.out + (size_t)m * a.ldo + 2 * u;
    h[0] = h0;
    h[1] = h1;
    if (a.stash) {
      float* s = a.stash + (size_t)m * a.ldo + 2 * u;
      s[0] = h0;
      s[1] = h1;
    }
    if (a.xbn_out) {  // the next projection's operand rows: h * gamma = hi + lo
      E[m * 128 + lr] = h0;
      E[m * 128 + lr + 1] = h1;
      T* hi = reinterpret_cast<T*>(a.xbn_out) + (size_t)m * a.ldo + 2 * u;
      T* lo = reinterpret_cast<T*>(a.xbn_out) + ((size_t)a.next_mp + m) * a.ldo + 2 * u;
      const float z0 = h0 * e_gamma[lr], z1 = h1 * e_gamma[lr + 1];
      const T a0 = Io<T>::from_f(z0), a1 = Io<T>::from_f(z1);
      hi[0] = a0;
      hi[1] = a1;
      lo[0] = Io<T>::from_f(z0 - Io<T>::to_f(a0));
      lo[1] = Io<T>::from_f(z1 - Io<T>::to_f(a1));
    }
    return;
  }
  const int half = a.hd >> 1;
  const int head = u / half, i = u - head * half;
  if (head < a.n_q + a.n_kv) {  // RoPE (rotate-half) on q and k
    const float c = E[m * 64 + i], s = E[MP * 64 + m * 64 + i];
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
    float* c = reinterpret_cast<float*>(is_k ? a.kcache : a.vcache);  // the KV cache is fp32
    const size_t base = ((((size_t)a.layer * a.n_pages + e_page[m]) * a.n_kv + kvh) * kPage + e_sidx[m]) * a.hd;
    c[base + i] = y0;
    c[base + i + half] = y1;
  }
}

constexpr int kMmaThreads = 192;  // warps 0-3 epilogue (TMEM lane quarters), 4 producer, 5 MMA issuer

// Items [w0, w1) of CTA b: an equal share of `total`.
__host__ __device__ __forceinline__ long long item_begin(long long total, int b, int G) { return total * b / G; }
// The CTA whose run holds item i.
__host__ __device__ __forceinline__ int item_cta(long long total, long long i, int G) {
  return (int)(((i + 1) * G - 1) / total);
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Completing CTA of a split tile: add the partial tiles of CTAs c0..c1 (its own included) into acc in
// CTA order, QBX tiles' loads in flight per round; rows m >= RV (and m >= M) are not read.  (Loading
// only a verify pass's valid rows, to fit twice the tiles in a round, measured no faster.)
template <int NT, int MP, int RV, int QBX>
__device__ __forceinline__ void merge_partials(float (&acc)[NT][MP], const float* part, long long total, int G,
                                               int t, int stages, int c0, int c1, int r, int M) {
  for (int q0 = c0; q0 <= c1; q0 += QBX) {
    float v[QBX][NT][RV];
#pragma unroll
    for (int qq = 0; qq < QBX; ++qq) {
      const int q = q0 + qq;
      if (q <= c1) {
        const int seg = (int)(item_begin(total, q, G) / stages) == t ? 0 : 1;
        const float* src = part + (((size_t)q * 2 + seg) * NT) * MP * 128;
#pragma unroll
        for (int u = 0; u < NT; ++u)
#pragma unroll
          for (int m = 0; m < RV; ++m) v[qq][u][m] = m < M ? __ldcg(src + ((size_t)u * MP + m) * 128 + r) : 0.f;
      }
    }
#pragma unroll
    for (int qq = 0; qq < QBX; ++qq)
      if (q0 + qq <= c1) {
#pragma unroll
        for (int u = 0; u < NT; ++u)
#pragma unroll
          for (int m = 0; m < RV; ++m) acc[u][m] += v[qq][u][m];
      }
  }
}

template <typename T, int MP, int NT>
__global__ void __launch_bounds__(kMmaThreads, 1)
    k_mma(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tx, MmaArgs a) {
  using L = MmaSmem<MP, NT>;
  constexpr int XT = L::XT, SB = L::kStage, S = L::kStages;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  float* C = reinterpret_cast<float*>(smem + S * SB);  // [NT][MP][128]
  // Epilogue inputs of the current tile, loaded while its MMAs run: residual rows (RESID) or RoPE cos | sin
  // (QKV) as [MP][128] floats, then per row the scale, cache page and slot in page.
  float* E = reinterpret_cast<float*>(smem + S * SB + L::kC);
  float* e_scale = E + (NT == 1 ? MP * 128 : 0);
  int* e_page = reinterpret_cast<int*>(e_scale + MP);
  int* e_sidx = e_page + MP;
  float* e_gamma = reinterpret_cast<float*>(e_sidx + 2 * MP);  // RESID: the next RMSNorm's gains of this tile
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * SB + L::kC + L::kE);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;   // [2] MMA -> epilogue
  uint64_t* acc_empty = acc_full + 2;  // [2] epilogue -> MMA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, b = blockIdx.x;
  const long long total = (long long)a.n_tiles * a.stages;
  const long long w0 = item_begin(total, b, G), w1 = item_begin(total, b + 1, G);
  const int t_first = (int)(w0 / a.stages), t_last = (int)((w1 - 1) / a.stages);
  const int F = a.ep.F;
  constexpr uint32_t kCols = tmem_pow2(2 * NT * 2 * MP);  // two accumulators of NT units of 2 * MP columns
  const bool bf16 = std::is_same<T, __nv_bfloat16>::value;

  griddep_launch();
  trace_mark(a.ep.trace, 0);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;
  const uint32_t stage_tx = (uint32_t)(NT * kWT + (a.int8 ? 1 : 2) * XT);

  if (warp == 4) {
    if (lane == 0) {
      // ---- producer: weight tiles of the first stages may be requested before the dependency wait
      auto load_w = [&](long long i, int slot) {
        const int t = (int)(i / a.stages), k = (int)(i - (long long)t * a.stages) * kBK;
        unsigned char* st = smem + slot * SB;
        tma_load_2d(st, &tw, k, t * 128, &full[slot]);
        if (NT == 2) tma_load_2d(st + kWT, &tw, k, F + t * 128, &full[slot]);
      };
      const int pre = (int)min((long long)S, w1 - w0);
      for (int i = 0; i < pre; ++i) {
        mbar_expect_tx(&full[i], stage_tx);
        load_w(w0 + i, i);
      }
      griddep_wait();
      for (long long i = w0; i < w1; ++i) {
        const int n = (int)(i - w0), slot = n % S;
        const int k = (int)(i % a.stages) * kBK;
        unsigned char* st = smem + slot * SB;
        if (n >= S) {
          if (!mbar_wait_bounded(&empty[slot], (uint32_t)(((n / S) - 1) & 1))) {
            ok = false;
            break;
          }
          mbar_expect_tx(&full[slot], stage_tx);
          load_w(i, slot);
        }
        tma_load_2d(st + NT * kWT, &tx, k, 0, &full[slot]);  // hi rows, then the lo rows (one box)
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      // ---- MMA issuer: segment j (the part of tile t_first + j in this CTA's run) into accumulator j & 1
      const uint32_t idesc = idesc_f16(a.int8 ? MP : 2 * MP, bf16);
      long long i = w0;
      for (int j = 0; ok && j <= t_last - t_first; ++j) {
        const int buf = j & 1;
        if (j >= 2 && !mbar_wait_bounded(&acc_empty[buf], (uint32_t)(((j >> 1) - 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const long long seg_end = min(w1, (long long)(t_first + j + 1) * a.stages);
        const uint32_t d0 = tmem + (uint32_t)(buf * NT * 2 * MP);
        for (bool first = true; i < seg_end; ++i, first = false) {
          const int n = (int)(i - w0), slot = n % S;
          if (!mbar_wait_bounded(&full[slot], (uint32_t)((n / S) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t base = smem_u32(smem + slot * SB);
          const uint32_t xhi = base + NT * kWT;  // hi rows, then (not int8) the lo rows: one B operand
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint32_t acc = (!first || kk > 0) ? 1u : 0u;
            const uint64_t bx = sdesc_sw128(xhi + kk * 32);
#pragma unroll
            for (int t = 0; t < NT; ++t)
              mma_f16(d0 + t * 2 * MP, sdesc_sw128(base + t * kWT + kk * 32), bx, idesc, acc);
          }
          mma_commit(&empty[slot]);
        }
        mma_commit(&acc_full[buf]);
      }
    }
  } else {
    // ---- epilogue warps 0-3: thread r holds weight row r of the tile (TMEM lane r).  The outputs it
    // writes may be read or written by earlier kernels of the stream: wait for them too.
    griddep_wait();
    trace_mark(a.ep.trace, 1);
    const int r = warp * 32 + lane;
    for (int j = 0; j <= t_last - t_first; ++j) {
      const int t = t_first + j, buf = j & 1;
      const long long s_a = max(w0, (long long)t * a.stages), s_b = min(w1, (long long)(t + 1) * a.stages);
      float acc[NT][MP];
      {  // epilogue inputs of tile t, overlapping its MMAs (the previous segment's epilogue is done with E)
        const int n0 = t * 128;
        if (r < a.M) {
          if (a.ep.ss_in) {  // RMSNorm handed off by the previous residual epilogue: finish it here
            float ss = 0.f;
            for (int q = 0; q < a.ep.ss_tiles; ++q) ss += a.ep.ss_in[q * 64 + r];
            e_scale[r] = 1.0f / sqrtf(ss / (float)a.K + a.ep.eps);
          } else {
            e_scale[r] = a.scale[r];
          }
          if (a.ep.epi == EPI_QKV) {
            const int slot = a.ep.desc->slot[a.ep.row0 + r];
            e_page[r] = a.ep.btab[slot / kPage];
            e_sidx[r] = slot % kPage;
          }
        }
        if (NT == 1 && a.ep.epi == EPI_RESID) {
          for (int idx = r; idx < a.M * 128; idx += 128) {
            const int m = idx >> 7, row = idx & 127;
            if (n0 + row < a.ep.N) E[idx] = a.ep.out[(size_t)m * a.ep.ldo + n0 + row];
          }
          if (a.ep.xbn_out && n0 + r < a.ep.N) e_gamma[r] = Io<T>::to_f(reinterpret_cast<const T*>(a.ep.gamma_next)[n0 + r]);
        } else if (NT == 1 && a.ep.epi == EPI_QKV) {
          const int half = a.ep.hd >> 1;
          for (int idx = r; idx < a.M * half; idx += 128) {
            const int m = idx / half, i = idx - m * half;
            const int pos = a.ep.desc->pos[a.ep.row0 + m];
            E[m * 64 + i] = a.ep.rope_cos[(size_t)pos * half + i];
            E[MP * 64 + m * 64 + i] = a.ep.rope_sin[(size_t)pos * half + i];
          }
        }
      }
      // warp-uniform outcome: tcgen05.ld is a warp-wide (.sync.aligned) instruction
      const bool got = __all_sync(0xffffffffu, mbar_wait_bounded(&acc_full[buf], (uint32_t)((j >> 1) & 1)));
      if (!got) ok = false;
      tc_fence_after();
      if (got) {
#pragma unroll
        for (int u = 0; u < NT; ++u)
#pragma unroll
          for (int c = 0; c < MP; c += acc_chunk<MP>()) {
            const uint32_t col = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)((buf * NT + u) * 2 * MP + c);
            tmem_acc<MP>(col, a.int8, &acc[u][c]);
          }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(&acc_empty[buf]);
      bool have = got;
      if (s_b - s_a < a.stages) {
        // a tile shared with other CTAs: store this segment's partial sums; the CTA completing the tile adds
        // the segments up in CTA order
        float* mine = a.part + (((size_t)b * 2 + (j == 0 ? 0 : 1)) * NT) * MP * 128;
#pragma unroll
        for (int u = 0; u < NT; ++u)
#pragma unroll
          for (int m = 0; m < MP; ++m) mine[((size_t)u * MP + m) * 128 + r] = acc[u][m];
        // the epilogue warps' stores are ordered before thread 0's release by the barrier (fence
        // cumulativity), and the completing CTA's acquire before its threads' loads by the next one
        epi_bar();
        if (threadIdx.x == 0) {
          asm volatile("fence.acq_rel.gpu;" ::: "memory");
          const int prev = atomicAdd(a.counters + t, (int)(s_b - s_a));
          s_last = prev + (int)(s_b - s_a) == a.stages;
          if (s_last) {
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
            a.counters[t] = 0;
          }
        }
        epi_bar();
        have = s_last != 0;
        if (have) {
#pragma unroll
          for (int u = 0; u < NT; ++u)
#pragma unroll
            for (int m = 0; m < MP; ++m) acc[u][m] = 0.f;
          const long long ta = (long long)t * a.stages;
          const int c0 = item_cta(total, ta, G), c1 = item_cta(total, ta + a.stages - 1, G);
          // partial tiles added in CTA order, 64 / (NT * MP) tiles' loads in flight at once
          merge_partials<NT, MP, MP, (64 / (NT * MP) > 0 ? 64 / (NT * MP) : 1)>(acc, a.part, total, G, t, a.stages,
                                                                               c0, c1, r, a.M);
        }
      }
      if (have) {
        // stage the tile [u][m][row] in shared memory, then the epilogue over (row, unit) pairs
#pragma unroll
        for (int u = 0; u < NT; ++u)
#pragma unroll
          for (int m = 0; m < MP; ++m) C[((size_t)u * MP + m) * 128 + r] = acc[u][m];
      }
      epi_bar();
      if (have) {
        const int n0 = t * 128;
        const int units = NT == 2 ? 128 : 64;
        const int u0 = NT == 2 ? n0 : n0 / 2;
        const int nu = n_units(a.ep);
        for (int idx = r; idx < a.M * units; idx += 128) {
          const int m = idx / units, u = u0 + (idx - m * units);
          if (u >= nu) continue;
          int r0, r1;
          unit_rows(a.ep, u, r0, r1);
          float y0, y1;
          if (NT == 2) {
            y0 = C[(size_t)m * 128 + (r0 - n0)];
            y1 = C[((size_t)MP + m) * 128 + (r1 - F - n0)];
          } else {
            y0 = C[(size_t)m * 128 + (r0 - n0)];
            y1 = C[(size_t)m * 128 + (r1 - n0)];
          }
          const float sc = e_scale[m];
          if (NT == 1 && (a.ep.epi == EPI_RESID || a.ep.epi == EPI_QKV))
            epi_staged<T, MP>(a.ep, m, u, y0 * sc, y1 * sc, n0, E, e_page, e_sidx, e_gamma);
          else
            epi_apply<T>(a.ep, m, u, y0 * sc, y1 * sc);
        }
      }
      if (NT == 1 && a.ep.ss_out) {  // this tile's sum of h^2 per row (E holds the updated rows)
        epi_bar();
        if (have)
          for (int m = warp; m < a.M; m += 4) {
            float ssq = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float v = E[m * 128 + lane + 32 * k];
              ssq = fmaf(v, v, ssq);
            }
            ssq = warp_sum(ssq);
            if (lane == 0) a.ep.ss_out[t * 64 + m] = ssq;
          }
      }
      epi_bar();  // C is reused by the next segment
    }
  }
  if (!ok && a.ep.err) atomicExch(a.ep.err, 2);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols) : "memory");
  trace_mark(a.ep.trace, 2);
}

// ---------------------------------------------------------------- split-K in a thread-block cluster

namespace cg = cooperative_groups;

template <int MP, int NT>
struct SplitSmem {
  static constexpr int XT = MP * kBK * 2;
  static constexpr int kStage = NT * kWT + 2 * XT;
  // epilogue inputs (as in k_mma) and per-row scale / cache page / slot; the partial tile [NT][MP][128]
  // that the cluster reads reuses the ring, which is idle once the accumulator is complete
  static constexpr int kE = NT == 1 ? MP * 128 * 4 + MP * 16 + 128 * 4 : MP * 16;
  static constexpr int kS0 = (kMmaSmemBudget - 2048 - kE) / kStage;
  static constexpr int kStages = kS0 > 8 ? 8 : kS0;
  static constexpr int kBars = (2 * kStages + 2) * 8 + 16;
  static constexpr int kBytes = 1024 + kStages * kStage + kE + kBars;
  static_assert(kStages * kStage >= NT * MP * 128 * 4, "the partial tile must fit the ring");
};

template <typename T, int MP, int NT>
__global__ void __launch_bounds__(kMmaThreads, 1)
    k_mma_split(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tx, MmaArgs a) {
  using L = SplitSmem<MP, NT>;
  constexpr int XT = L::XT, SB = L::kStage, S = L::kStages;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  float* C = reinterpret_cast<float*>(smem);  // [NT][MP][128] partial tile, after the last MMA
  float* E = reinterpret_cast<float*>(smem + S * SB);
  float* e_scale = E + (NT == 1 ? MP * 128 : 0);
  int* e_page = reinterpret_cast<int*>(e_scale + MP);
  int* e_sidx = e_page + MP;
  float* e_gamma = reinterpret_cast<float*>(e_sidx + 2 * MP);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * SB + L::kE);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 2);
  cg::cluster_group cluster = cg::this_cluster();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nc = (int)cluster.num_blocks(), rank = (int)cluster.block_rank();
  const int t = blockIdx.x / nc;  // the output tile (pair) of this cluster
  const int k0 = rank * a.stages / nc, k1 = (rank + 1) * a.stages / nc;  // this rank's K stages
  const int F = a.ep.F;
  constexpr uint32_t kCols = tmem_pow2(NT * 2 * MP);  // NT units of 2 * MP columns
  const bool bf16 = std::is_same<T, __nv_bfloat16>::value;

  griddep_launch();
  trace_mark(a.ep.trace, 0);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(&acc_full[0], 1);
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;
  const uint32_t stage_tx = (uint32_t)(NT * kWT + (a.int8 ? 1 : 2) * XT);
  const int n_items = k1 - k0;

  if (warp == 4) {
    if (lane == 0 && n_items > 0) {
      // ---- producer: the first weight stages are requested before the dependency wait
      auto load_w = [&](int k, int slot) {
        unsigned char* st = smem + slot * SB;
        tma_load_2d(st, &tw, k * kBK, t * 128, &full[slot]);
        if (NT == 2) tma_load_2d(st + kWT, &tw, k * kBK, F + t * 128, &full[slot]);
      };
      const int pre = min(S, n_items);
      for (int i = 0; i < pre; ++i) {
        mbar_expect_tx(&full[i], stage_tx);
        load_w(k0 + i, i);
      }
      griddep_wait();
      for (int n = 0; n < n_items; ++n) {
        const int slot = n % S, k = k0 + n;
        unsigned char* st = smem + slot * SB;
        if (n >= S) {
          if (!mbar_wait_bounded(&empty[slot], (uint32_t)(((n / S) - 1) & 1))) {
            ok = false;
            break;
          }
          mbar_expect_tx(&full[slot], stage_tx);
          load_w(k, slot);
        }
        tma_load_2d(st + NT * kWT, &tx, k * kBK, 0, &full[slot]);  // hi rows, then the lo rows (one box)
      }
    }
  } else if (warp == 5) {
    if (lane == 0 && n_items > 0) {
      // ---- MMA issuer: this rank's K stages into one accumulator
      const uint32_t idesc = idesc_f16(a.int8 ? MP : 2 * MP, bf16);
      for (int n = 0; n < n_items; ++n) {
        const int slot = n % S;
        if (!mbar_wait_bounded(&full[slot], (uint32_t)((n / S) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t base = smem_u32(smem + slot * SB);
        const uint32_t xhi = base + NT * kWT;  // hi rows, then (not int8) the lo rows: one B operand
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint32_t acc = (n > 0 || kk > 0) ? 1u : 0u;
          const uint64_t bx = sdesc_sw128(xhi + kk * 32);
#pragma unroll
          for (int u = 0; u < NT; ++u)
            mma_f16(tmem + u * 2 * MP, sdesc_sw128(base + u * kWT + kk * 32), bx, idesc, acc);
        }
        mma_commit(&empty[slot]);
      }
      mma_commit(&acc_full[0]);  // arrives once every MMA issued above has completed
    }
  } else {
    // ---- epilogue warps 0-3: thread r holds weight row r of the tile (TMEM lane r)
    griddep_wait();
    trace_mark(a.ep.trace, 1);
    const int r = warp * 32 + lane;
    const int n0 = t * 128;
    if (r < a.M) {  // epilogue inputs, loaded while the MMAs run
      if (a.ep.ss_in) {  // RMSNorm handed off by the previous residual epilogue: finish it here
        float ss = 0.f;
        for (int q = 0; q < a.ep.ss_tiles; ++q) ss += a.ep.ss_in[q * 64 + r];
        e_scale[r] = 1.0f / sqrtf(ss / (float)a.K + a.ep.eps);
      } else {
        e_scale[r] = a.scale[r];
      }
      if (a.ep.epi == EPI_QKV) {
        const int slot = a.ep.desc->slot[a.ep.row0 + r];
        e_page[r] = a.ep.btab[slot / kPage];
        e_sidx[r] = slot % kPage;
      }
    }
    if (NT == 1 && a.ep.epi == EPI_RESID) {
      for (int idx = r; idx < a.M * 128; idx += 128) {
        const int m = idx >> 7, row = idx & 127;
        if (n0 + row < a.ep.N) E[idx] = a.ep.out[(size_t)m * a.ep.ldo + n0 + row];
      }
      if (a.ep.xbn_out && n0 + r < a.ep.N) e_gamma[r] = Io<T>::to_f(reinterpret_cast<const T*>(a.ep.gamma_next)[n0 + r]);
    } else if (NT == 1 && a.ep.epi == EPI_QKV) {
      const int half = a.ep.hd >> 1;
      for (int idx = r; idx < a.M * half; idx += 128) {
        const int m = idx / half, i = idx - m * half;
        const int pos = a.ep.desc->pos[a.ep.row0 + m];
        E[m * 64 + i] = a.ep.rope_cos[(size_t)pos * half + i];
        E[MP * 64 + m * 64 + i] = a.ep.rope_sin[(size_t)pos * half + i];
      }
    }
    float acc[NT][MP];
    bool got = n_items > 0;
    if (got) {  // warp-uniform: tcgen05.ld is a warp-wide instruction
      got = __all_sync(0xffffffffu, mbar_wait_bounded(&acc_full[0], 0u));
      if (!got) ok = false;
    }
    tc_fence_after();
    if (got) {
#pragma unroll
      for (int u = 0; u < NT; ++u)
#pragma unroll
        for (int c = 0; c < MP; c += acc_chunk<MP>()) {
          const uint32_t col = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(u * 2 * MP + c);
          tmem_acc<MP>(col, a.int8, &acc[u][c]);
        }
    } else {
#pragma unroll
      for (int u = 0; u < NT; ++u)
#pragma unroll
        for (int m = 0; m < MP; ++m) acc[u][m] = 0.f;
    }
    tc_fence_before();
    fence_proxy_async();  // the ring was last written by TMA and read by the tensor cores
    epi_bar();  // every epilogue thread is past the accumulator wait: the ring is idle from here on
#pragma unroll
    for (int u = 0; u < NT; ++u)
#pragma unroll
      for (int m = 0; m < MP; ++m) C[((size_t)u * MP + m) * 128 + r] = acc[u][m];
  }
  cluster.sync();  // every rank's partial tile is written and visible to the cluster
  if (warp < 4) {
    const int r = warp * 32 + lane;
    const int n0 = t * 128;
    const int units = NT == 2 ? 128 : 64;  // output units of the tile
    const int u_lo = rank * units / nc, u_hi = (rank + 1) * units / nc, cnt = u_hi - u_lo;
    const int ug0 = NT == 2 ? n0 : n0 / 2;  // first unit of the tile
    const int nu = n_units(a.ep);
    const float* cr[8];  // every rank's partial tile (this rank's through its own shared-memory window)
#pragma unroll
    for (int q = 0; q < 8; ++q) cr[q] = q < nc ? (q == rank ? C : cluster.map_shared_rank(C, (unsigned)q)) : C;
    for (int idx = r; idx < a.M * cnt; idx += 128) {
      const int m = idx / cnt, u = ug0 + u_lo + (idx - m * cnt);
      if (u >= nu) continue;
      int r0, r1;
      unit_rows(a.ep, u, r0, r1);
      const int o0 = m * 128 + (r0 - n0), o1 = (NT == 2 ? MP * 128 : 0) + m * 128 + (NT == 2 ? r1 - F - n0 : r1 - n0);
      float v0[8], v1[8];  // all ranks' loads in flight at once, then added in rank order
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < nc) {
          v0[q] = cr[q][o0];
          v1[q] = cr[q][o1];
        }
      float y0 = 0.f, y1 = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < nc) {
          y0 += v0[q];
          y1 += v1[q];
        }
      const float sc = e_scale[m];
      if (NT == 1 && (a.ep.epi == EPI_RESID || a.ep.epi == EPI_QKV))
        epi_staged<T, MP>(a.ep, m, u, y0 * sc, y1 * sc, n0, E, e_page, e_sidx, e_gamma);
      else
        epi_apply<T>(a.ep, m, u, y0 * sc, y1 * sc);
    }
  }
  // this CTA reads no other rank's shared memory from here on; its own must outlive the others' reads
  cluster.barrier_arrive();
  if (warp < 4) {
    const int units = NT == 2 ? 128 : 64;
    const int u_lo = rank * units / nc, u_hi = (rank + 1) * units / nc;
    if (NT == 1 && a.ep.ss_out) {  // this rank's share of the tile's sum of h^2 per row (E holds its rows)
      epi_bar();
      const int f_lo = 2 * u_lo, f_hi = 2 * u_hi;
      for (int m = warp; m < a.M; m += 4) {
        float ssq = 0.f;
        for (int f = f_lo + lane; f < f_hi; f += 32) {
          const float v = E[m * 128 + f];
          ssq = fmaf(v, v, ssq);
        }
        ssq = warp_sum(ssq);
        if (lane == 0) a.ep.ss_out[(t * nc + rank) * 64 + m] = ssq;
      }
    }
  }
  if (!ok && a.ep.err) atomicExch(a.ep.err, 2);
  tc_fence_before();
  cluster.barrier_wait();  // no CTA leaves (freeing its shared memory) while another rank still reads it
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols) : "memory");
  trace_mark(a.ep.trace, 2);
}

// ---------------------------------------------------------------- host side

namespace {

// The driver's tensor-map encoder, found through the runtime (no link-time dependency on libcuda).
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool encode_2d(CUtensorMap* map, const void* base, int fp16, uint64_t inner, uint64_t outer, uint32_t box_inner,
               uint32_t box_outer) {
  return encode_rows_2d(map, base, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, inner,
                        outer, box_inner, box_outer);
}

}  // namespace

bool encode_rows_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, size_t elem_bytes, uint64_t inner,
                    uint64_t outer, uint32_t box_inner, uint32_t box_outer) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * elem_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

// Clusters of c CTAs (c = 1..8) of k_mma_split<T, MP, NT> that can be resident at once, from the occupancy
// calculator (index [fp16][mp_slot(MP)][NT - 1][c]); 0 = unknown (that size is not used).
constexpr int mp_slot(int mp) { return mp == 8 ? 0 : mp / 16; }
int g_split_max[2][5][2][9];

template <typename T, int MP, int NT>
void fill_split_max() {
  int* out = g_split_max[std::is_same<T, __half>::value ? 1 : 0][mp_slot(MP)][NT - 1];
  for (int c = 1; c <= 8; ++c) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(c);
    cfg.blockDim = dim3(kMmaThreads);
    cfg.dynamicSmemBytes = SplitSmem<MP, NT>::kBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k_mma_split<T, MP, NT>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
    out[c] = n;
  }
}

// Ranks per cluster of the split-K kernel for a matrix of n_tiles output tiles (pairs) and `stages` K
// stages, or 0 for stream-K: the most ranks (<= 8, <= stages) with n_tiles * c <= SMs whose clusters all
// fit at once, provided that keeps at least 60 % of the SMs streaming (fewer tiles than that: stream-K; the 8B
// QKV projection's 48 tiles x 2 ranks = 96 CTAs took the 7-row verify pass from 3.68 to 3.33 ms against
// stream-K on all 152 SMs).  mode 1 drops the 60 % rule, mode 2 always answers stream-K.
int split_ways(int n_tiles, int stages, int sms, const int* maxc, int mode) {
  if (n_tiles > sms || mode == 2) return 0;
  for (int c = 8; c >= 1; --c)
    if (n_tiles * c <= sms && c <= stages && maxc[c] >= n_tiles)
      return (mode == 1 || 10 * n_tiles * c >= 6 * sms) ? c : 0;
  return 0;
}

template <typename T, int MP, int NT>
int split_of(int n_rows, int K, int sms, int mode) {
  return split_ways((n_rows + 127) / 128, (K + kBK - 1) / kBK, sms,
                    g_split_max[std::is_same<T, __half>::value ? 1 : 0][mp_slot(MP)][NT - 1], mode);
}

template <typename T, int MP, int NT>
bool run_mma(const LinearArgs& ep, const MmaScratch& sc, int* counters, int sms, cudaStream_t st) {
  using L = MmaSmem<MP, NT>;
  const int K = ep.K, M = ep.M;
  const int n_rows = NT == 2 ? ep.F : ep.N;
  if (K % 8 || (ep.epi == EPI_QKV && 128 % ep.hd)) return false;
  if (ep.xb_ready && ep.int8) return false;  // handed-off operands are hi/lo pairs, never int8 codes
  MmaArgs a{};
  a.M = M;
  a.K = K;
  a.n_tiles = (n_rows + 127) / 128;
  a.stages = (K + kBK - 1) / kBK;
  if (a.n_tiles > 4096) return false;  // counters
  const int ways = split_of<T, MP, NT>(n_rows, K, sms, ep.mma_mode);
  const long long total = (long long)a.n_tiles * a.stages;
  const int G = (int)std::min<long long>(sms, total);
  if (!ways && (size_t)G * 2 * NT * MP * 128 * 4 > sc.part_bytes) return false;
  const void* xb = ep.xb_ready ? ep.xb_ready : sc.xb;
  float* scale = ep.xb_ready ? const_cast<float*>(sc.ones) : sc.scale;
  float* part = sc.part;
  a.int8 = ep.int8;
  a.scale = scale;
  a.part = part;
  a.counters = counters;
  a.ep = ep;

  CUtensorMap tw, tx;
  const int fp16 = std::is_same<T, __half>::value;
  if (!encode_2d(&tw, ep.W, fp16, (uint64_t)K, (uint64_t)ep.N, kBK, 128)) return false;
  // the activation box: the hi rows and the lo rows below them ([2][MP][K]) in one copy; int8 codes: MP rows
  if (!encode_2d(&tx, xb, fp16, (uint64_t)K, (uint64_t)2 * MP, kBK, ep.int8 ? MP : 2 * MP)) return false;

  if (!ep.xb_ready) {
    PrepArgs p{};
    p.X = ep.X;
    p.ldx = ep.ldx;
    p.M = M;
    p.Mpad = MP;
    p.K = K;
    p.gamma = ep.gamma;
    p.eps = ep.eps;
    p.int8 = ep.int8;
    p.xb = sc.xb;
    p.scale = scale;
    p.trace = ep.trace_prep;
    launch_ex(k_act_prep<T>, dim3(MP), dim3(256), 0, st, p);
  }
  if (ways) {  // one tile per cluster of `ways` CTAs
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ways;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(a.n_tiles * ways);
    cfg.blockDim = dim3(kMmaThreads);
    cfg.dynamicSmemBytes = SplitSmem<MP, NT>::kBytes;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = g_pdl ? 2 : 1;
    g_launches += 1;
    return cudaLaunchKernelEx(&cfg, k_mma_split<T, MP, NT>, tw, tx, a) == cudaSuccess;
  }
  launch_ex(k_mma<T, MP, NT>, dim3(G), dim3(kMmaThreads), (size_t)L::kBytes, st, tw, tx, a);
  return true;
}

template <typename T, int MP>
bool run_mma_nt(const LinearArgs& a, const MmaScratch& sc, int* counters, int sms, cudaStream_t st) {
  return a.epi == EPI_SWIGLU ? run_mma<T, MP, 2>(a, sc, counters, sms, st) : run_mma<T, MP, 1>(a, sc, counters, sms, st);
}

template <typename T>
bool dispatch(const LinearArgs& a, const MmaScratch& sc, int* counters, int sms, cudaStream_t st) {
  // int8 codes fill only MP of the MMA's columns, which must be at least 16
  const int mp = a.int8 && mma_rows_pad(a.M) < 16 ? 16 : mma_rows_pad(a.M);
  switch (mp) {
    case 8:
      return run_mma_nt<T, 8>(a, sc, counters, sms, st);
    case 16:
      return run_mma_nt<T, 16>(a, sc, counters, sms, st);
    case 32:
      return run_mma_nt<T, 32>(a, sc, counters, sms, st);
    case 48:
      return run_mma_nt<T, 48>(a, sc, counters, sms, st);
    default:
      return run_mma_nt<T, 64>(a, sc, counters, sms, st);
  }
}

template <typename T, int MP, int NT>
bool set_attr1() {
  static_assert(MmaSmem<MP, NT>::kStages >= 2 && SplitSmem<MP, NT>::kStages >= 2, "ring too shallow");
  const bool ok = cudaFuncSetAttribute(k_mma<T, MP, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       MmaSmem<MP, NT>::kBytes) == cudaSuccess &&
                  cudaFuncSetAttribute(k_mma_split<T, MP, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SplitSmem<MP, NT>::kBytes) == cudaSuccess;
  if (ok) fill_split_max<T, MP, NT>();
  return ok;
}

template <typename T, int MP>
bool set_attr() {
  return set_attr1<T, MP, 1>() && set_attr1<T, MP, 2>();
}

}  // namespace

bool init_kernels() {
  static std::once_flag once;
  static bool ok = false;
  std::call_once(once, [] {
    ok = init_linear_kernels() && init_attention_kernels();
    ok = ok && set_attr<__nv_bfloat16, 8>() && set_attr<__nv_bfloat16, 16>() && set_attr<__nv_bfloat16, 32>() &&
         set_attr<__nv_bfloat16, 48>() && set_attr<__nv_bfloat16, 64>();
    ok = ok && set_attr<__half, 8>() && set_attr<__half, 16>() && set_attr<__half, 32>() && set_attr<__half, 48>() &&
         set_attr<__half, 64>();
  });
  return ok;
}

int mma_ss_slots(int n_rows, int K, int M, int fp16, int sms, int mode) {
  int ways = 0;
  const int mp = mma_rows_pad(M);
  if (fp16) {
    ways = mp == 8    ? split_of<__half, 8, 1>(n_rows, K, sms, mode)
         : mp == 16 ? split_of<__half, 16, 1>(n_rows, K, sms, mode)
         : mp == 32 ? split_of<__half, 32, 1>(n_rows, K, sms, mode)
         : mp == 48 ? split_of<__half, 48, 1>(n_rows, K, sms, mode) : split_of<__half, 64, 1>(n_rows, K, sms, mode);
  } else {
    ways = mp == 8    ? split_of<__nv_bfloat16, 8, 1>(n_rows, K, sms, mode)
         : mp == 16 ? split_of<__nv_bfloat16, 16, 1>(n_rows, K, sms, mode)
         : mp == 32 ? split_of<__nv_bfloat16, 32, 1>(n_rows, K, sms, mode)
         : mp == 48 ? split_of<__nv_bfloat16, 48, 1>(n_rows, K, sms, mode)
                    : split_of<__nv_bfloat16, 64, 1>(n_rows, K, sms, mode);
  }
  return (n_rows + 127) / 128 * (ways ? ways : 1);
}

int mma_split_ways(int n_rows, int K, int M, int nt, int fp16, int sms, int mode) {
  const int mp = mma_rows_pad(M);
#define SSD_WAYS(T, MPV) (nt == 2 ? split_of<T, MPV, 2>(n_rows, K, sms, mode) : split_of<T, MPV, 1>(n_rows, K, sms, mode))
  if (fp16)
    return mp == 8 ? SSD_WAYS(__half, 8) : mp == 16 ? SSD_WAYS(__half, 16) : mp == 32 ? SSD_WAYS(__half, 32)
         : mp == 48 ? SSD_WAYS(__half, 48) : SSD_WAYS(__half, 64);
  return mp == 8 ? SSD_WAYS(__nv_bfloat16, 8) : mp == 16 ? SSD_WAYS(__nv_bfloat16, 16)
       : mp == 32 ? SSD_WAYS(__nv_bfloat16, 32) : mp == 48 ? SSD_WAYS(__nv_bfloat16, 48) : SSD_WAYS(__nv_bfloat16, 64);
#undef SSD_WAYS
}

int mma_rows_pad(int M) { return M <= 8 ? 8 : M <= 16 ? 16 : M <= 32 ? 32 : M <= 48 ? 48 : 64; }

bool launch_mma(const LinearArgs& a, int fp16, const MmaScratch& sc, int* counters, int sms, cudaStream_t st) {
  if (a.M < 2 || a.M > 64) return false;
  return fp16 ? dispatch<__half>(a, sc, counters, sms, st) : dispatch<__nv_bfloat16>(a, sc, counters, sms, st);
}

}  // namespace ssd

extern "C" void ssd_streamk_split(int64_t total, int G, int b, int64_t i, int64_t* begin, int* cta) {
  if (total <= 0 || G <= 0) return;
  if (begin) *begin = ssd::item_begin(total, b, G);
  if (cta) *cta = ssd::item_cta(total, i, G);
}
