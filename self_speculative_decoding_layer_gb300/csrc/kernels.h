// Host-side launch interface of libssd's kernels (internal; not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace ssd {

// Kernels launched by this process's launchers (host-side count, for statistics).
extern thread_local long long g_launches;

enum Epi { EPI_QKV = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_LOGITS = 3 };

// y = W x for every input row, with a fused prologue on x and a fused epilogue on y.
//   prologue: optional RMSNorm (gamma != null) then optional per-token int8
//             quantization of the (normalised) row.
//   epilogue: EPI_QKV    rotate q, k (RoPE), write q (fp32) and k, v (16-bit cache)
//             EPI_RESID  out[m][r] += y (residual add); optional stash copy
//             EPI_SWIGLU out[m][j] = SiLU(y_gate[j]) * y_up[j]   (W rows: gate, then up)
//             EPI_LOGITS out[m][r] = y
struct LinearArgs {
  const void* W;  // [N, K] 16-bit, row-major
  int N, K;
  const float* X;  // [M, ldx]
  int ldx;
  int M;
  int row0;  // index of X's row 0 in the pass (for the descriptor)
  const void* gamma;
  float eps;
  int int8;
  int epi;
  float* out;
  int ldo;
  float* stash;  // RESID: copy of the updated row, [M, ldo] (may be null)
  // QKV
  void* kcache;
  void* vcache;
  const int* btab;
  int n_pages, layer, n_q, n_kv, hd;
  const float* rope_cos;
  const float* rope_sin;
  const PassDesc* desc;
  int F;  // SWIGLU: ffn width
  // stream-K GEMV: partial sums of row pairs split between two warps, their
  // arrival counters (zero between launches) and the device error flag
  float* sk_part;
  int* sk_cnt;
  int* err;
  // L2 prefetch of the weights the pass reads next (issued when this CTA's share is done)
  const void* pf;
  size_t pf_bytes;
  unsigned long long* trace;       // timeline slot (SSD_OPT_TRACE) or null
  unsigned long long* trace_prep;  // input preparation kernel of the tensor-core path (tracing only)
  // Tensor-core path, operand hand-off: xb_ready = this projection's 16-bit operand rows, already written
  // by the kernel that produced X ([2][Mpad][K]: hi rows then lo rows), so no preparation kernel runs;
  // xb_next (SwiGLU epilogue) = where to write the next projection's operand rows ([2][next_mp][F]).
  const void* xb_ready;
  void* xb_next;
  int next_mp;
  // RMSNorm hand-off (tensor-core path).  RESID epilogue: also write the next projection's operand rows
  // as hi/lo of h * gamma_next ([2][next_mp][ldo]) and each tile's per-row sum of h^2 (ss_out[tile*64 + m]).
  // Consumer (with xb_ready): 1/rms of row m from ss_in (ss_tiles tiles, added in tile order), applied as
  // the row scale of its result.
  void* xbn_out;
  const void* gamma_next;
  float* ss_out;
  const float* ss_in;
  int ss_tiles;
  // Draft exit gate (&DevState::draft_live) of a later draft forward, or null: the kernel returns right
  // after its dependency wait once drafting has stopped.
  const int* gate;
  // Work distribution of the tensor-core path: 0 = by shape (split-K in a cluster or stream-K), 1 = split-K
  // wherever the tiles fit the SMs, 2 = stream-K (1 and 2 are set by the test library only).
  int mma_mode;
};

void launch_gemv_rs(const LinearArgs& a, int fp16, int sms, cudaStream_t st);    // M == 1, register stream-K
#ifdef SSD_CROSSCHECK
// Cross-check kernels of the test library (not in the product library).
void launch_linear_rows(const LinearArgs& a, int fp16, cudaStream_t st);        // any M, CUDA cores
void launch_gemv(const LinearArgs& a, int fp16, cudaStream_t st);               // M == 1, register streaming
void launch_gemv_bulk(const LinearArgs& a, int fp16, int sms, cudaStream_t st);  // M == 1, TMA-bulk stream-K
#endif

// Programmatic dependent launch for every kernel of a pass (set per context before capture).
extern thread_local bool g_pdl;

// Launch with the programmatic-stream-serialization attribute when g_pdl is
// set: the kernel may start while its predecessor drains, so every kernel
// calls griddep_wait() before touching anything a predecessor writes.
template <typename... KArgs, typename... Args>
inline void launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = g_pdl ? 1 : 0;
  g_launches += 1;
  cudaLaunchKernelEx(&cfg, kern, args...);
}
// 2D tensor map over a row-major [outer][inner] matrix of elem_bytes-sized
// elements, boxes of box_outer rows x box_inner elements, 128-byte swizzle.
bool encode_rows_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, size_t elem_bytes, uint64_t inner,
                    uint64_t outer, uint32_t box_inner, uint32_t box_outer);
// Device scratch of the tensor-core path: operand rows written by the preparation kernel, its per-row
// scales, a row of ones (scales of handed-off operands) and the stream-K partial tiles.
struct MmaScratch {
  void* xb;
  float* scale;
  const float* ones;
  float* part;
  size_t part_bytes;
};
int mma_rows_pad(int M);  // operand rows of an M-row projection (8, 16, 32, 48 or 64; int8 codes: at least 16)
// Per-row sum-of-squares slots a residual projection of n_rows outputs writes for the RMSNorm hand-off
// (one per output tile, or per tile and rank when the split-K kernel runs it); the consumer's ss_tiles.
int mma_ss_slots(int n_rows, int K, int M, int fp16, int sms, int mma_mode);
// Ranks per output tile (pair, nt = 2) of the split-K kernel for an M-row projection of n_rows outputs, or 0
// when the stream-K kernel runs it (16-bit operands).
int mma_split_ways(int n_rows, int K, int M, int nt, int fp16, int sms, int mma_mode);
bool launch_mma(const LinearArgs& a, int fp16, const MmaScratch& sc, int* tile_counters, int sms,
                cudaStream_t st);  // tcgen05 path; false if the shape is unsupported

struct AttnArgs {
  const PassDesc* desc;
  const float* q;  // [R, Hq*hd]
  const void* kcache;
  const void* vcache;
  const int* btab;
  int n_pages, layer, n_q, n_kv, hd;
  float* out;      // [R, Hq*hd]
  int rows;
  int n_split;     // key splits = cluster size (1, 2, 4 or 8)
  int qb;          // queries (of one KV head's group) per CTA, 1..32: grid z = ceil(rows * group / qb)
  // optional operand hand-off to the output projection: hi/lo 16-bit copies of out ([2][next_mp][n_q*hd],
  // fp16 if xb_fp16 else bf16)
  void* xb_next;
  int next_mp, xb_fp16;
  int max_keys;    // most keys any launch of this (captured) kernel sees: sizes the tile ring
  int ring_cap;    // most bytes of tile ring (0: the whole shared-memory budget)
  int n_slots;     // set by launch_attention
  int* err;        // device error flag (a TMA wait ran out), or null
  // L2 prefetch of the weights the pass reads next (HBM is otherwise idle during attention)
  const void* pf;
  size_t pf_bytes;
  unsigned long long* trace;
  const int* gate;  // draft exit gate, as in LinearArgs
  // early != 0: prefix tiles whose keys all lie below *committed (the committed length) are copied into
  // the ring before the dependency wait.  Only for launches in a pass replayed as one graph: no earlier
  // pass is still running then, and no kernel of the pass writes a slot below the committed length.
  const int* committed;
  int early;
  // After the dependency wait, while HBM is otherwise idle: an L2 prefetch of the first head_bytes of each of
  // rows rows (stride bytes apart) of the matrix the layer streams after the output projection (gate/up),
  // set when each of its CTAs starts its K loop at column 0 of its tiles (one tile pair per CTA), so that
  // every CTA finds its first stages in L2.  Null: none.
  const char* head_pf;
  int head_rows, head_stride, head_bytes;
};
// kv_type: element type of the caches, 0 bf16, 1 fp16, 2 fp32.  False if the
// arguments are out of range, a tensor map cannot be encoded or the launch fails.
bool launch_attention(const AttnArgs& a, int kv_type, cudaStream_t st);
// Store a row descriptor given by value into device memory (the standalone attention's scratch).
bool launch_store_desc(const PassDesc& d, PassDesc* out, cudaStream_t st);
bool init_attention_kernels();
// Grid of an attention launch that sees at most max_keys keys: queries per CTA (*qb: 4, 8, 16 or 32) and
// key splits (*n_split = cluster size: 1, 2, 4 or 8) for rows x group queries per KV head; kv_type, hd and
// ring_cap as for launch_attention / AttnArgs (they set the ring and so the clusters that fit at once).
void attention_layout(int max_keys, int rows, int group, int n_kv, int kv_type, int hd, int ring_cap, int* qb,
                      int* n_split);

// One-time kernel attribute set-up (outside any stream capture); false if a CUDA call failed.
bool init_kernels();

}  // namespace ssd
