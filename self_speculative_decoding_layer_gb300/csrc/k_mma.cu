// Tensor-core (tcgen05) projections for 2..64 input rows: the verify pass
// (K+1 rows), tree verification (N+1 rows), the CLaSp DP rows and prefill
// chunks.
//
// Y[M, N] = X[M, K] W[N, K]^T is computed as D[128, Mpad] = W_tile X^T
// ("swap AB"): 128 weight rows fill the MMA's M dimension and the few input
// rows are its N dimension (Mpad = M rounded up to 16).  The input rows are
// first prepared by k_act_prep -- the same RMSNorm / int8 arithmetic as the
// CUDA-core kernels -- and stored as 16-bit operands: a hi/lo pair
// (x = hi + lo, both bf16 or both fp16 like the weights) whose two MMAs keep
// the activation at close to fp32 precision, or the int8 codes (exact in 16
// bits) with a per-row scale.  Each CTA streams its weight tile over a K
// range through a 4-stage TMA (SWIZZLE_128B) + mbarrier ring; one thread
// issues tcgen05.mma into a TMEM accumulator; a K range split over several
// CTAs is summed by the last one in a fixed order; the epilogue is the one of
// the CUDA-core kernels (RoPE + KV write, residual, SwiGLU, logits).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace ssd {

bool init_linear_kernels();

constexpr int kNS = 4;              // pipeline stages
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
  griddep_wait();
  const int m = blockIdx.x;
  T* hi = reinterpret_cast<T*>(a.xb) + (size_t)m * a.K;
  T* lo = reinterpret_cast<T*>(a.xb) + ((size_t)a.Mpad + m) * a.K;
  if (m >= a.M) {  // padding rows are zero
    for (int k = threadIdx.x; k < a.K; k += blockDim.x) {
      hi[k] = Io<T>::from_f(0.f);
      lo[k] = Io<T>::from_f(0.f);
    }
    if (threadIdx.x == 0) a.scale[m] = 0.f;
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

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
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

// ---------------------------------------------------------------- the GEMM kernel

struct MmaArgs {
  int M, K;
  int n_tiles;  // 128-row weight tiles (SwiGLU: gate/up tile pairs)
  int splits;   // CTAs per tile along K
  int stages;   // K stages of kBK elements
  int swiglu, int8;
  const float* scale;
  float* part;    // split-K partials [n_tiles][splits][nt][Mpad][128]
  int* counters;  // [n_tiles], zero between launches
  LinearArgs ep;  // epilogue targets
};

template <int MP>
struct MmaSmem {
  static constexpr int XT = MP * kBK * 2;  // one activation operand tile (hi or lo)
  static constexpr __host__ __device__ int stage(int nt) { return nt * kWT + 2 * XT; }
  static constexpr __host__ __device__ int bytes(int nt) { return 1024 + kNS * stage(nt) + (2 * kNS + 2) * 8 + 16; }
};

template <typename T, int MP>
__global__ void __launch_bounds__(128, 1)
    k_mma(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tx, MmaArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  constexpr int XT = MmaSmem<MP>::XT;
  const int nt = a.swiglu ? 2 : 1;
  const int SB = MmaSmem<MP>::stage(nt);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kNS * SB);
  uint64_t* empty = full + kNS;
  uint64_t* done = empty + kNS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x / a.splits, sp = blockIdx.x - tile * a.splits;
  const int s_lo = (int)((long long)sp * a.stages / a.splits);
  const int s_hi = (int)((long long)(sp + 1) * a.stages / a.splits);
  const int ns = s_hi - s_lo;
  const int n0 = tile * 128;
  const int F = a.ep.F;
  const uint32_t ncols = (uint32_t)(nt * MP <= 32 ? 32 : (nt * MP <= 64 ? 64 : 128));
  const bool bf16 = sizeof(T) == 2 && !std::is_same<T, __half>::value;

  griddep_launch();
  trace_mark(a.ep.trace, 0);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    for (int i = 0; i < kNS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(done, 1);
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;
  const uint32_t stage_tx = (uint32_t)(nt * kWT + (a.int8 ? 1 : 2) * XT);

  if (warp == 0 && lane == 0) {
    // ---- producer: weight tiles may be requested before the dependency wait
    const int pre = ns < kNS ? ns : kNS;
    for (int i = 0; i < pre; ++i) {
      unsigned char* st = smem + i * SB;
      mbar_expect_tx(&full[i], stage_tx);
      const int k = (s_lo + i) * kBK;
      tma_load_2d(st, &tw, k, n0, &full[i]);
      if (nt == 2) tma_load_2d(st + kWT, &tw, k, F + n0, &full[i]);
    }
    griddep_wait();
    for (int i = 0; i < ns && ok; ++i) {
      const int slot = i % kNS;
      unsigned char* st = smem + slot * SB;
      const int k = (s_lo + i) * kBK;
      if (i >= kNS) {
        if (!mbar_wait_bounded(&empty[slot], (uint32_t)(((i / kNS) - 1) & 1))) {
          ok = false;
          break;
        }
        mbar_expect_tx(&full[slot], stage_tx);
        tma_load_2d(st, &tw, k, n0, &full[slot]);
        if (nt == 2) tma_load_2d(st + kWT, &tw, k, F + n0, &full[slot]);
      }
      tma_load_2d(st + nt * kWT, &tx, k, 0, &full[slot]);                     // hi rows
      if (!a.int8) tma_load_2d(st + nt * kWT + XT, &tx, k, MP, &full[slot]);  // lo rows
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    griddep_wait();
    const uint32_t idesc = idesc_f16(MP, bf16);
    for (int i = 0; i < ns; ++i) {
      const int slot = i % kNS;
      if (!mbar_wait_bounded(&full[slot], (uint32_t)((i / kNS) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t base = smem_u32(smem + slot * SB);
      const uint32_t xhi = base + nt * kWT, xlo = xhi + XT;
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
        const uint64_t bh = sdesc_sw128(xhi + kk * 32), bl = sdesc_sw128(xlo + kk * 32);
        for (int t = 0; t < nt; ++t) {
          const uint64_t ad = sdesc_sw128(base + t * kWT + kk * 32);
          mma_f16(tmem + t * MP, ad, bh, idesc, acc);
          if (!a.int8) mma_f16(tmem + t * MP, ad, bl, idesc, 1u);
        }
      }
      mma_commit(&empty[slot]);
    }
    mma_commit(done);
  }
  griddep_wait();
  trace_mark(a.ep.trace, 1);
  __syncwarp();

  // ---- epilogue: warp w holds weight rows 32w .. 32w+31 of the tile
  if (!mbar_wait_bounded(done, 0)) ok = false;
  tc_fence_after();
  float acc[2][MP];
  const int r = warp * 32 + lane;
  for (int t = 0; t < nt; ++t)
#pragma unroll
    for (int c = 0; c < MP; c += 16)
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(t * MP + c), &acc[t][c]);

  __shared__ int s_last;
  bool last = true;
  if (a.splits > 1) {
    float* mine = a.part + (((size_t)tile * a.splits + sp) * nt) * MP * 128;
    for (int t = 0; t < nt; ++t)
#pragma unroll
      for (int m = 0; m < MP; ++m) mine[((size_t)t * MP + m) * 128 + r] = acc[t][m];
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const int prev = atomicAdd(a.counters + tile, 1);
      s_last = prev == a.splits - 1;
      if (s_last) {
        __threadfence();
        a.counters[tile] = 0;
      }
    }
    __syncthreads();
    last = s_last != 0;
    if (last) {  // sum the splits in a fixed order
      for (int t = 0; t < nt; ++t)
#pragma unroll
        for (int m = 0; m < MP; ++m) acc[t][m] = 0.f;
      for (int q = 0; q < a.splits; ++q) {
        const float* src = a.part + (((size_t)tile * a.splits + q) * nt) * MP * 128;
        for (int t = 0; t < nt; ++t)
#pragma unroll
          for (int m = 0; m < MP; ++m) acc[t][m] += __ldcg(src + ((size_t)t * MP + m) * 128 + r);
      }
    }
  }
  if (last) {
    // stage the tile [t][m][row] in shared memory (the pipeline buffers are idle now)
    float* C = reinterpret_cast<float*>(smem);
    for (int t = 0; t < nt; ++t)
#pragma unroll
      for (int m = 0; m < MP; ++m) C[((size_t)t * MP + m) * 128 + r] = acc[t][m];
    __syncthreads();
    const int units = a.swiglu ? 128 : 64;
    const int u0 = a.swiglu ? n0 : n0 / 2;
    const int nu = n_units(a.ep);
    for (int idx = threadIdx.x; idx < a.M * units; idx += blockDim.x) {
      const int m = idx / units, u = u0 + (idx - m * units);
      if (u >= nu) continue;
      int r0, r1;
      unit_rows(a.ep, u, r0, r1);
      float y0, y1;
      if (a.swiglu) {
        y0 = C[(size_t)m * 128 + (r0 - n0)];
        y1 = C[((size_t)MP + m) * 128 + (r1 - F - n0)];
      } else {
        y0 = C[(size_t)m * 128 + (r0 - n0)];
        y1 = C[(size_t)m * 128 + (r1 - n0)];
      }
      const float s = a.scale[m];
      epi_apply<T>(a.ep, m, u, y0 * s, y1 * s);
    }
  }
  if (!ok && threadIdx.x == 0 && a.ep.err) atomicExch(a.ep.err, 2);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
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

template <typename T, int MP>
bool run_mma(const LinearArgs& ep, void* scratch, size_t scratch_bytes, int* counters, int sms, cudaStream_t st) {
  const int K = ep.K, M = ep.M;
  const bool swiglu = ep.epi == EPI_SWIGLU;
  const int nt = swiglu ? 2 : 1;
  const int n_rows = swiglu ? ep.F : ep.N;
  if (K % 8 || (ep.epi == EPI_QKV && 128 % ep.hd)) return false;
  // scratch: [xb: 2 x MP x K 16-bit][scale: 64 floats][partials]
  char* sc = reinterpret_cast<char*>(scratch);
  const size_t xb_bytes = ((size_t)2 * MP * K * 2 + 1023) & ~(size_t)1023;
  void* xb = sc;
  float* scale = reinterpret_cast<float*>(sc + xb_bytes);
  float* part = reinterpret_cast<float*>(sc + xb_bytes + 1024);
  const size_t part_cap = scratch_bytes - xb_bytes - 1024;

  MmaArgs a{};
  a.M = M;
  a.K = K;
  a.n_tiles = (n_rows + 127) / 128;
  a.stages = (K + kBK - 1) / kBK;
  a.swiglu = swiglu;
  a.int8 = ep.int8;
  a.scale = scale;
  a.part = part;
  a.counters = counters;
  a.ep = ep;
  int splits = (sms + a.n_tiles - 1) / a.n_tiles;
  if (splits > a.stages) splits = a.stages;
  if (splits < 1) splits = 1;
  while (splits > 1 && (size_t)a.n_tiles * splits * nt * MP * 128 * 4 > part_cap) --splits;
  if (a.n_tiles > 4096) return false;  // counters
  a.splits = splits;

  CUtensorMap tw, tx;
  const int fp16 = std::is_same<T, __half>::value;
  if (!encode_2d(&tw, ep.W, fp16, (uint64_t)K, (uint64_t)ep.N, kBK, 128)) return false;
  if (!encode_2d(&tx, xb, fp16, (uint64_t)K, (uint64_t)2 * MP, kBK, MP)) return false;

  PrepArgs p{};
  p.X = ep.X;
  p.ldx = ep.ldx;
  p.M = M;
  p.Mpad = MP;
  p.K = K;
  p.gamma = ep.gamma;
  p.eps = ep.eps;
  p.int8 = ep.int8;
  p.xb = xb;
  p.scale = scale;
  launch_ex(k_act_prep<T>, dim3(MP), dim3(256), 0, st, p);
  const size_t smem = (size_t)MmaSmem<MP>::bytes(nt);
  launch_ex(k_mma<T, MP>, dim3(a.n_tiles * a.splits), dim3(128), smem, st, tw, tx, a);
  return true;
}

template <typename T>
bool dispatch(const LinearArgs& a, void* scratch, size_t bytes, int* counters, int sms, cudaStream_t st) {
  if (a.M <= 16) return run_mma<T, 16>(a, scratch, bytes, counters, sms, st);
  if (a.M <= 32) return run_mma<T, 32>(a, scratch, bytes, counters, sms, st);
  if (a.M <= 48) return run_mma<T, 48>(a, scratch, bytes, counters, sms, st);
  return run_mma<T, 64>(a, scratch, bytes, counters, sms, st);
}

template <typename T, int MP>
bool set_attr() {
  return cudaFuncSetAttribute(k_mma<T, MP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              MmaSmem<MP>::bytes(2)) == cudaSuccess;
}

}  // namespace

bool init_kernels() {
  bool ok = init_linear_kernels() && init_attention_kernels();
  ok &= set_attr<__nv_bfloat16, 16>() && set_attr<__nv_bfloat16, 32>() && set_attr<__nv_bfloat16, 48>() &&
        set_attr<__nv_bfloat16, 64>();
  ok &= set_attr<__half, 16>() && set_attr<__half, 32>() && set_attr<__half, 48>() && set_attr<__half, 64>();
  return ok;
}

bool launch_mma(const LinearArgs& a, int fp16, void* scratch, size_t scratch_bytes, int* counters, int sms,
                cudaStream_t st) {
  if (a.M < 2 || a.M > 64) return false;
  return fp16 ? dispatch<__half>(a, scratch, scratch_bytes, counters, sms, st)
              : dispatch<__nv_bfloat16>(a, scratch, scratch_bytes, counters, sms, st);
}

}  // namespace ssd
