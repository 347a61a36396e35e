// Pass set-up, greedy argmax / top-2, acceptance + rollback, KV compaction,
// and the CLaSp DP step / backtrack kernels.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "misc.h"

namespace ssd {

// ---------------------------------------------------------------- pass set-up

// Builds the PassDesc of the pass from the device state, records each row's
// token and writes the rows' embeddings E[token] (fp32) into h (and the
// layer-0 stash row).  One CTA per row; CTA 0 / thread 0 writes the
// descriptor.
template <typename T>
__global__ void k_begin(BeginArgs a) {
  griddep_launch();
  trace_mark(a.trace, 0);
  griddep_wait();
  trace_mark(a.trace, 1);
  const int r = blockIdx.x;
  DevState* st = a.st;
  const int step = a.step >= 0 ? a.step : *reinterpret_cast<const volatile int*>(&st->draft_n);
  if (a.kind == BEGIN_DRAFT && a.exit_k) {
    if (step == 0) {  // open the gate; drafts not reached before the exit stay -1, which no argmax equals
      int* drafts = const_cast<int*>(a.tok);
      for (int j = threadIdx.x; j < a.exit_k; j += blockDim.x) drafts[j] = -1;
      if (threadIdx.x == 0) {
        st->draft_live = 1;
        st->draft_n = 0;
      }
    } else if (!gate_open(&st->draft_live)) {
      return;
    }
  }
  const int t = st->t;
  int tok = 0;
  if (a.kind != BEGIN_DP) {
    if (a.kind == BEGIN_DRAFT) {
      tok = step == 0 ? st->pending : a.tok[step - 1];
    } else if (a.kind == BEGIN_EXPAND) {
      const int node = a.exp_node[st->exp_idx];
      tok = node == 0 ? st->pending : a.tok[node];
    } else if (a.kind == BEGIN_TREE) {
      tok = r == 0 ? st->pending : a.tok[r];
    } else {
      tok = (a.first_pending && r == 0) ? st->pending : a.tok[a.tok_offset + r - a.first_pending];
    }
    // a verify row past a draft exit carries token -1: it is embedded as token 0 (its result is never used);
    // an id past the vocabulary cannot come from a correct pass: it is flagged and row 0 read instead
    if (tok >= a.vocab) {
      if (threadIdx.x == 0) atomicExch(&st->err, kDevErrToken);
      tok = 0;
    }
    const T* e = reinterpret_cast<const T*>(a.E) + (size_t)(tok < 0 ? 0 : tok) * a.d;
    float* h = a.h + (size_t)r * a.ldh;
    float* s0 = a.stash0 ? a.stash0 + (size_t)r * a.ldh : nullptr;
    // the embedding row in 16-byte pieces, every load issued before the first is used (a row is one
    // random HBM location: a load-use chain per element would pay its latency d / blockDim times)
    constexpr int U = 4;
    for (int base = threadIdx.x * 8; base < a.d; base += U * 8 * (int)blockDim.x) {
      uint4 raw[U];
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const int k = base + j * 8 * (int)blockDim.x;
        if (k + 8 <= a.d) raw[j] = *reinterpret_cast<const uint4*>(e + k);
      }
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const int k = base + j * 8 * (int)blockDim.x;
        if (k + 8 <= a.d) {
          float v[8];
          Io<T>::unpack8(raw[j], v);
          *reinterpret_cast<float4*>(h + k) = make_float4(v[0], v[1], v[2], v[3]);
          *reinterpret_cast<float4*>(h + k + 4) = make_float4(v[4], v[5], v[6], v[7]);
          if (s0) {
            *reinterpret_cast<float4*>(s0 + k) = make_float4(v[0], v[1], v[2], v[3]);
            *reinterpret_cast<float4*>(s0 + k + 4) = make_float4(v[4], v[5], v[6], v[7]);
          }
        } else {
          for (int q = k; q < a.d; ++q) {  // ragged end (d not a multiple of 8)
            const float v = Io<T>::to_f(e[q]);
            h[q] = v;
            if (s0) s0[q] = v;
          }
        }
      }
    }
  }
  if (threadIdx.x == 0) {
    PassDesc* d = a.desc;
    if (a.row_tok) a.row_tok[r] = tok;
    switch (a.kind) {
      case BEGIN_CAUSAL:
        d->pos[r] = t + r;
        d->slot[r] = t + r;
        d->mask[r] = (r == 63) ? ~0ull : ((1ull << (r + 1)) - 1ull);
        if (r == 0) {
          d->prefix = t;
          d->base = t;
        }
        break;
      case BEGIN_DRAFT:
        d->pos[0] = t + step;
        d->slot[0] = t + step;
        d->mask[0] = 1ull;
        d->prefix = t + step;
        d->base = t + step;
        break;
      case BEGIN_TREE:
        d->pos[r] = t + a.depth[r];
        d->slot[r] = t + r;
        d->mask[r] = a.anc[r];
        if (r == 0) {
          d->prefix = t;
          d->base = t;
        }
        break;
      case BEGIN_EXPAND: {
        const int node = a.exp_node[st->exp_idx];
        d->pos[0] = t + a.depth[node];
        d->slot[0] = t + node;
        d->mask[0] = a.anc[node];
        d->prefix = t;
        d->base = t;
        break;
      }
      case BEGIN_DP:
        d->pos[r] = st->tgt_pos;
        d->slot[r] = t + r;  // scratch slots past the committed length
        d->mask[r] = 1ull << r;
        if (r == 0) {
          d->prefix = st->tgt_pos;
          d->base = t;
        }
        break;
    }
    if (r == 0) d->rows = a.rows;
  }
  trace_mark(a.trace, 2);
}

void launch_begin(const BeginArgs& a, int fp16, cudaStream_t st) {
  if (fp16)
    launch_ex(k_begin<__half>, dim3(a.rows), dim3(256), 0, st, a);
  else
    launch_ex(k_begin<__nv_bfloat16>, dim3(a.rows), dim3(256), 0, st, a);
}

// ---------------------------------------------------------------- argmax / top-2

struct Top2 {
  float v1, v2;
  int i1, i2;
  float z;  // draft exit: sum over the part of exp(x - v1)
};

__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// A NaN logit counts as -inf, so every row yields ids inside the vocabulary.
__device__ __forceinline__ void top2_push(Top2& t, float v, int i) {
  if (v != v) v = -INFINITY;
  if (better(v, i, t.v1, t.i1)) {
    t.v2 = t.v1;
    t.i2 = t.i1;
    t.v1 = v;
    t.i1 = i;
  } else if (better(v, i, t.v2, t.i2)) {
    t.v2 = v;
    t.i2 = i;
  }
}

__device__ __forceinline__ Top2 top2_merge(Top2 a, const Top2& b) {
  top2_push(a, b.v1, b.i1);
  top2_push(a, b.v2, b.i2);
  return a;
}

// Softmax normaliser in (max, sum of exp(x - max)) form: merge (mo, zo) into (m, z).
// Float addition is commutative, so both lanes of a butterfly step get the same value.
__device__ __forceinline__ void lse_merge(float& m, float& z, float mo, float zo) {
  const float M = fmaxf(m, mo);
  if (M == -INFINITY) return;
  z = z * __expf(m - M) + zo * __expf(mo - M);
  m = M;
}

__device__ __forceinline__ void lse_warp(float& m, float& z) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, o), zo = __shfl_xor_sync(0xffffffffu, z, o);
    lse_merge(m, z, mo, zo);
  }
}

// Greedy longest-prefix acceptance over a chain (parents == null) or a tree.
// Walks from the root to the child whose token equals the full model's
// argmax at the current node; the bonus is the argmax where the walk stops.
// Updates committed length (rollback of the rest), pending token, the DP
// target row, statistics and the output buffer.  One thread; am may have been
// written by other CTAs of the same launch (read through L2).
__device__ void accept_walk(DevState* st, const int* row_tok, const int* parents, const int* am, int n_rows,
                            int* out_tokens) {
  const int t = st->t;
  int cur = 0, n = 0;
  st->path[0] = 0;
  while (true) {
    const int want = __ldcg(am + cur);
    int nxt = -1;
    if (parents == nullptr) {
      if (cur + 1 < n_rows && row_tok[cur + 1] == want) nxt = cur + 1;
    } else {
      for (int c = cur + 1; c < n_rows; ++c)
        if (parents[c] == cur && row_tok[c] == want) {
          nxt = c;
          break;
        }
    }
    if (nxt < 0) break;
    cur = nxt;
    st->path[++n] = cur;
  }
  const int bonus = __ldcg(am + cur);
  st->n_acc = n;
  st->bonus = bonus;
  st->last_path_len = n + 1;
  st->tgt_row = cur;
  st->tgt_pos = t + n;
  st->t = t + n + 1;
  st->pending = bonus;
  st->cycles += 1;
  st->accepted += n;
  st->hist[n] += 1;
  int nd = 0;  // drafts verified: chain rows past a draft exit hold -1
  for (int r = 1; r < n_rows; ++r) nd += parents != nullptr || row_tok[r] >= 0;
  st->drafted += nd;
  if (out_tokens) {
    for (int i = 1; i <= n; ++i) {
      if (st->gen_count < st->gen_cap) out_tokens[st->gen_count] = row_tok[st->path[i]];
      st->gen_count += 1;
    }
    if (st->gen_count < st->gen_cap) out_tokens[st->gen_count] = bonus;
    st->gen_count += 1;
  }
}

// Greedy token (ties -> lowest id) and runner-up of each logits row.
// kArgBlocks CTAs share a row: each reduces its slice to a top-two pair
// (eight independent loads in flight per thread), stores it, and the CTA
// that completes the row merges the pairs.  Value descending, then id
// ascending, is a total order, so the result does not depend on which CTA
// finishes last.  With a draft exit the softmax normaliser of the row is
// reduced alongside (per thread, per warp by butterfly, per CTA in warp
// order, per row over the CTAs' parts by butterfly): a fixed order, so p1
// is reproducible run to run.
constexpr int kArgBlocks = 32;

__device__ __forceinline__ Top2 top2_warp(Top2 t) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Top2 u;
    u.v1 = __shfl_xor_sync(0xffffffffu, t.v1, o);
    u.v2 = __shfl_xor_sync(0xffffffffu, t.v2, o);
    u.i1 = __shfl_xor_sync(0xffffffffu, t.i1, o);
    u.i2 = __shfl_xor_sync(0xffffffffu, t.i2, o);
    t = top2_merge(t, u);
  }
  return t;
}

__global__ void __launch_bounds__(256) k_argmax(const float* logits, int V, int ld, int* out1, int* out2, Top2* part,
                                                int* cnt, ArgmaxExit ex, AcceptArgs acc) {
  griddep_launch();
  griddep_wait();
  DevState* st = ex.st;
  if (st && !ex.dyn && ex.step > 0 && !gate_open(&st->draft_live)) return;
  const bool want_p = st != nullptr;
  // the draft's index: fixed, or the loop's count (changed only by this launch's last CTA, at its end)
  const int step = (st && ex.dyn) ? *reinterpret_cast<const volatile int*>(&st->draft_n) : ex.step;
  __shared__ Top2 s[8];
  __shared__ float s_m[8], s_z[8];
  __shared__ int s_last;
  const int row = blockIdx.y, blk = blockIdx.x, nb = gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* x = logits + (size_t)row * ld;
  const int per = (V + nb - 1) / nb;
  const int b0 = blk * per, b1 = min(V, b0 + per);
  Top2 t{-INFINITY, -INFINITY, 0x7fffffff, 0x7fffffff, 0.f};
  float m = -INFINITY, z = 0.f;  // this thread's max and sum of exp(x - max)
  for (int base = b0 + threadIdx.x; base < b1; base += 8 * 256) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = base + j * 256 < b1 ? x[base + j * 256] : -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (base + j * 256 < b1) top2_push(t, v[j], base + j * 256);
    if (want_p) {
      float mx = m;
#pragma unroll
      for (int j = 0; j < 8; ++j) mx = fmaxf(mx, v[j]);
      if (mx > m) {
        z = m == -INFINITY ? 0.f : z * __expf(m - mx);
        m = mx;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (base + j * 256 < b1) z += __expf(v[j] - m);
    }
  }
  t = top2_warp(t);
  if (want_p) lse_warp(m, z);
  if (lane == 0) {
    s[warp] = t;
    s_m[warp] = m;
    s_z[warp] = z;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    Top2 r = s[0];
    float rm = s_m[0], rz = s_z[0];
    for (int w = 1; w < 8; ++w) {
      r = top2_merge(r, s[w]);
      lse_merge(rm, rz, s_m[w], s_z[w]);
    }
    r.z = rz;  // rm == r.v1: both are the exact maximum of the slice
    part[(size_t)row * nb + blk] = r;
    __threadfence();
    s_last = atomicAdd(cnt + row, 1) == nb - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  Top2 r{-INFINITY, -INFINITY, 0x7fffffff, 0x7fffffff, 0.f};
  float rm = -INFINITY, rz = 0.f;
  if (threadIdx.x < 32) {
    for (int b = lane; b < nb; b += 32) {
      const Top2* q = part + (size_t)row * nb + b;
      Top2 u;
      u.v1 = __ldcg(&q->v1);
      u.v2 = __ldcg(&q->v2);
      u.i1 = __ldcg(&q->i1);
      u.i2 = __ldcg(&q->i2);
      r = top2_merge(r, u);
      if (want_p) lse_merge(rm, rz, u.v1, __ldcg(&q->z));
    }
    r = top2_warp(r);
    if (want_p) lse_warp(rm, rz);
    if (lane == 0) {
      out1[ex.dyn ? step : row] = r.i1;
      if (out2) out2[row] = r.i2;
      cnt[row] = 0;
      if (want_p) {
        const float p1 = 1.0f / rz;  // the top-1 term is exp(0) = 1, so rz >= 1
        const bool go_on = !(p1 < ex.thr);
        st->draft_p1[step] = p1;
        st->draft_n = step + 1;
        if (!go_on) st->draft_live = 0;
        if (ex.has_cond) cudaGraphSetConditional(ex.cond, (go_on && step + 1 < ex.k) ? 1u : 0u);
      }
      if (acc.st) {  // verify: the CTA that completes the last row accepts
        __threadfence();
        if (atomicAdd(acc.rows_done, 1) == (int)gridDim.y - 1) {
          __threadfence();
          *acc.rows_done = 0;
          accept_walk(acc.st, acc.row_tok, acc.parents, out1, acc.n_rows, acc.out_tokens);
        }
      }
    }
  }
}

// Vertical cascade: the higher draft level checked the lower level's k drafts (row r of its pass
// predicts the token after draft r-1; row 0 follows the pending token).  Keep the longest prefix it
// agrees with, replace the first draft it rejects by its own prediction and mark the rest -1, so the
// target's fixed (k+1)-row verify sees the higher level's drafts.
__global__ void k_draft_accept(const int* am, int* drafts, int k) {
  griddep_launch();
  griddep_wait();
  int n = 0;
  while (n < k && am[n] == drafts[n]) ++n;
  if (n < k) {
    drafts[n] = am[n];
    for (int j = n + 1; j < k; ++j) drafts[j] = -1;
  }
}

void launch_draft_accept(const int* am, int* drafts, int k, cudaStream_t s) {
  launch_ex(k_draft_accept, dim3(1), dim3(1), 0, s, am, drafts, k);
}

__global__ void k_draft_reset(DevState* st, int* drafts, int k) {
  griddep_launch();
  griddep_wait();
  for (int j = threadIdx.x; j < k; j += blockDim.x) drafts[j] = -1;
  if (threadIdx.x == 0) {
    st->draft_live = 1;
    st->draft_n = 0;
  }
}

void launch_draft_reset(DevState* st, int* drafts, int k, cudaStream_t s) {
  launch_ex(k_draft_reset, dim3(1), dim3(64), 0, s, st, drafts, k);
}

void launch_argmax(const float* logits, int rows, int V, int ld, int* out1, int* out2, void* part, int* cnt,
                   cudaStream_t st, ArgmaxExit ex, AcceptArgs acc) {
  launch_ex(k_argmax, dim3(kArgBlocks, rows), dim3(256), 0, st, logits, V, ld, out1, out2,
            reinterpret_cast<Top2*>(part), cnt, ex, acc);
}

size_t argmax_part_bytes(int rows) { return (size_t)rows * kArgBlocks * sizeof(Top2); }

// ---------------------------------------------------------------- commit / accept

// After a prefill chunk or an AR step: advance the committed length by `rows`
// and, if `take`, make argmax[0] the pending token (and append it to the
// output buffer when there is one).  The last row becomes the DP target.
__global__ void k_advance(DevState* st, int rows, const int* am, int take, int* out_tokens) {
  griddep_launch();
  griddep_wait();
  const int t = st->t;
  st->tgt_row = rows - 1;
  st->tgt_pos = t + rows - 1;
  st->t = t + rows;
  if (take) {
    st->pending = am[0];
    if (out_tokens && st->gen_count < st->gen_cap) out_tokens[st->gen_count] = am[0];
    st->gen_count += 1;
  }
}

void launch_advance(DevState* st, int rows, const int* am, int take, int* out_tokens, cudaStream_t s) {
  launch_ex(k_advance, dim3(1), dim3(1), 0, s, st, rows, am, take, out_tokens);
}

// Move the accepted tree path's K/V (all layers) from slot t0 + path[i] to
// slot t0 + i.  Grid: (layers, kv heads); destinations never overlap a later
// source because path[i] >= i and path is increasing.
template <typename T>
__global__ void k_compact(const DevState* st, T* kc, T* vc, const int* btab, int n_pages, int n_kv, int hd) {
  griddep_launch();
  griddep_wait();
  const int n = st->n_acc;
  const int t0 = st->t - n - 1;
  const int layer = blockIdx.x, kvh = blockIdx.y;
  for (int i = 1; i <= n; ++i) {
    const int src = t0 + st->path[i], dst = t0 + i;
    if (src == dst) continue;
    const size_t si = kv_index(layer, src, kvh, 0, btab, n_pages, n_kv, hd);
    const size_t di = kv_index(layer, dst, kvh, 0, btab, n_pages, n_kv, hd);
    for (int d = threadIdx.x; d < hd; d += blockDim.x) {
      kc[di + d] = kc[si + d];
      vc[di + d] = vc[si + d];
    }
    __syncthreads();
  }
}

void launch_compact(const DevState* st, void* kc, void* vc, const int* btab, int n_pages, int n_layers, int n_kv,
                    int hd, int fp16, cudaStream_t s) {
  (void)fp16;  // the context's KV cache is fp32
  dim3 grid(n_layers, n_kv);
  launch_ex(k_compact<float>, dim3(grid), dim3(128), 0, s, st, (float*)kc, (float*)vc, btab, n_pages, n_kv, hd);
}

// Store the top-2 continuation of the current DyTC expansion as the tokens of
// the node's two children (child id 0 = absent) and advance the expansion index.
__global__ void k_store_children(DevState* st, int* tree_tok, const int* child0, const int* child1, const int* am1,
                                 const int* am2) {
  griddep_launch();
  griddep_wait();
  const int e = st->exp_idx;
  if (child0[e] > 0) tree_tok[child0[e]] = am1[0];
  if (child1[e] > 0) tree_tok[child1[e]] = am2[0];
  st->exp_idx = e + 1;
}

void launch_store_children(DevState* st, int* tree_tok, const int* c0, const int* c1, const int* am1, const int* am2,
                           cudaStream_t s) {
  launch_ex(k_store_children, dim3(1), dim3(1), 0, s, st, tree_tok, c0, c1, am1, am2);
}

// ---------------------------------------------------------------- CLaSp DP

// The DP kernels hold a row in registers: every thread takes float4 elements tid, tid + blockDim, ... of it,
// kDpU of them at most (rows up to kDpU * 4 * blockDim floats; longer rows are read again to be stored).
// Sums are float per thread and per warp (rows of at most a few thousand elements, well inside the
// 2e-3 the DP values are compared to), and only the last few operations of a decision run in double, on
// one thread: FP64 throughput is a small fraction of FP32 here.
constexpr int kDpThreads = 256, kDpU = 8;

__device__ __forceinline__ float dot4(const float4& x, const float4& y) {
  return fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, x.w * y.w)));
}

template <typename T>
struct alignas(8) Pack4 {
  T v[4];
};

// Store element group i4 of the state chosen for DP column j: the state table row, and when the next
// layer runs (h set) its pass row r, plus for a tensor-core next layer (xb set) the QKV operand rows as
// 16-bit hi/lo of state * gamma (the consumer applies 1/rms from the row's sum of squares).
template <typename T>
__device__ __forceinline__ void dp_emit(int i4, const float4& v, float* state_row, float* h_row, T* hi_row, T* lo_row,
                                        const T* gamma) {
  if (state_row) reinterpret_cast<float4*>(state_row)[i4] = v;
  if (h_row) reinterpret_cast<float4*>(h_row)[i4] = v;
  if (hi_row) {
    const Pack4<T> g = reinterpret_cast<const Pack4<T>*>(gamma)[i4];
    const float z[4] = {v.x * Io<T>::to_f(g.v[0]), v.y * Io<T>::to_f(g.v[1]), v.z * Io<T>::to_f(g.v[2]),
                        v.w * Io<T>::to_f(g.v[3])};
    Pack4<T> h, l;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      h.v[e] = Io<T>::from_f(z[e]);
      l.v[e] = Io<T>::from_f(z[e] - Io<T>::to_f(h.v[e]));
    }
    reinterpret_cast<Pack4<T>*>(hi_row)[i4] = h;
    reinterpret_cast<Pack4<T>*>(lo_row)[i4] = l;
  }
}

// Block sum of NQ floats per thread; the totals, in double, on thread 0 only.
template <int NQ>
__device__ __forceinline__ void dp_block_sum(float (&acc)[NQ], double (&tot)[NQ]) {
  __shared__ float sh[kDpThreads / 32][NQ];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], o);
    if (lane == 0) sh[warp][q] = acc[q];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      tot[q] = 0.0;
      for (int w = 0; w < kDpThreads / 32; ++w) tot[q] += (double)sh[w][q];
    }
  }
}

// Initial state: state(0, 0) = the target's embedding row (stash layer 0), also the first layer's pass row.
template <typename T>
__global__ void __launch_bounds__(kDpThreads) k_dp_init(const DevState* st, const float* stash, int d, float* states,
                                                        float* val, unsigned char* back, float* h0, void* xb0,
                                                        float* ss0, const void* gamma0, int mp0) {
  griddep_launch();
  griddep_wait();
  const float* g0 = stash + (size_t)st->tgt_row * d;
  const int d4 = d >> 2;
  float acc[1] = {0.f};
  for (int i4 = threadIdx.x; i4 < d4; i4 += kDpThreads) {
    const float4 v = reinterpret_cast<const float4*>(g0)[i4];
    acc[0] += dot4(v, v);
    T* hi = xb0 ? reinterpret_cast<T*>(xb0) : nullptr;
    dp_emit<T>(i4, v, states, h0, hi, hi ? hi + (size_t)mp0 * d : nullptr, reinterpret_cast<const T*>(gamma0));
  }
  double tot[1];
  dp_block_sum<1>(acc, tot);
  if (threadIdx.x == 0) {
    if (xb0) ss0[0] = (float)tot[0];
    val[0] = 1.0f;
    back[0] = 0;
  }
}

void launch_dp_init(const DevState* st, const float* stash, int d, float* states, float* val, unsigned char* back,
                    float* h0, void* xb0, float* ss0, const void* gamma0, int mp0, int fp16, cudaStream_t s) {
  if (fp16)
    launch_ex(k_dp_init<__half>, dim3(1), dim3(kDpThreads), 0, s, st, stash, d, states, val, back, h0, xb0, ss0,
              gamma0, mp0);
  else
    launch_ex(k_dp_init<__nv_bfloat16>, dim3(1), dim3(kDpThreads), 0, s, st, stash, d, states, val, back, h0, xb0,
              ss0, gamma0, mp0);
}

// One DP layer step (layer i = 1..L).  CTA per j in [lo_i, hi_i]:
//   keep = layer-i output of state(i-1, j)   (pass row j - lo_prev), if j <= hi_prev
//   skip = state(i-1, j-1),                   if j-1 >= lo_prev
// state(i, j) = the one with the larger cos(., g_i); a tie keeps.  Every load of the three rows is in
// flight before the sums; the chosen row is stored from registers.
template <typename T>
__global__ void __launch_bounds__(kDpThreads) k_dp_step(DPStepArgs a) {
  griddep_launch();
  griddep_wait();
  __shared__ int s_keep;
  __shared__ float s_sumsq;
  const int j = a.lo + blockIdx.x;
  const int d4 = a.d >> 2;
  const float4* g = reinterpret_cast<const float4*>(a.stash_i + (size_t)a.st->tgt_row * a.d);
  const bool has_keep = j >= a.lo_prev && j <= a.hi_prev;
  const bool has_skip = (j - 1) >= a.lo_prev && (j - 1) <= a.hi_prev;
  const float4* keep = has_keep ? reinterpret_cast<const float4*>(a.h + (size_t)(j - a.lo_prev) * a.ldh) : nullptr;
  const float4* skip = has_skip ? reinterpret_cast<const float4*>(a.states_old + (size_t)(j - 1) * a.d) : nullptr;
  // |g|^2, |keep|^2, keep.g, |skip|^2, skip.g
  float acc[5] = {0.f, 0.f, 0.f, 0.f, 0.f};
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 kv[kDpU], sv[kDpU];
  const bool in_regs = d4 <= kDpU * kDpThreads;
  for (int base = threadIdx.x; base < d4; base += kDpU * kDpThreads) {
    float4 gv[kDpU];
#pragma unroll
    for (int u = 0; u < kDpU; ++u) {
      const int i4 = base + u * kDpThreads;
      const bool in = i4 < d4;
      gv[u] = in ? g[i4] : zero;
      kv[u] = in && keep ? keep[i4] : zero;
      sv[u] = in && skip ? skip[i4] : zero;
    }
#pragma unroll
    for (int u = 0; u < kDpU; ++u) {
      acc[0] += dot4(gv[u], gv[u]);
      acc[1] += dot4(kv[u], kv[u]);
      acc[2] += dot4(kv[u], gv[u]);
      acc[3] += dot4(sv[u], sv[u]);
      acc[4] += dot4(sv[u], gv[u]);
    }
  }
  double tot[5];
  dp_block_sum<5>(acc, tot);
  if (threadIdx.x == 0) {
    const double gg = tot[0], kk = tot[1], kg = tot[2], ss = tot[3], sg = tot[4];
    const double ck = keep ? kg / sqrt(kk * gg) : -2.0;
    const double cs = skip ? sg / sqrt(ss * gg) : -2.0;
    const bool take_keep = keep && ck >= cs;
    s_keep = take_keep ? 1 : 0;
    s_sumsq = (float)(take_keep ? kk : ss);
    a.val[(size_t)a.i * a.ncol + j] = (float)(take_keep ? ck : cs);
    a.back[(size_t)a.i * a.ncol + j] = take_keep ? 0 : 1;
  }
  __syncthreads();
  const bool take_keep = s_keep != 0;
  const int r = j - a.lo;
  float* state_row = a.states_new + (size_t)j * a.d;
  float* h_row = a.next_h ? a.next_h + (size_t)r * a.d : nullptr;
  T* hi = a.next_h && a.next_xb ? reinterpret_cast<T*>(a.next_xb) + (size_t)r * a.d : nullptr;
  T* lo = hi ? reinterpret_cast<T*>(a.next_xb) + ((size_t)a.next_mp + r) * a.d : nullptr;
  const T* gamma = reinterpret_cast<const T*>(a.next_gamma);
  if (in_regs) {
#pragma unroll
    for (int u = 0; u < kDpU; ++u) {
      const int i4 = threadIdx.x + u * kDpThreads;
      if (i4 < d4) dp_emit<T>(i4, take_keep ? kv[u] : sv[u], state_row, h_row, hi, lo, gamma);
    }
  } else {
    const float4* src = take_keep ? keep : skip;
    for (int i4 = threadIdx.x; i4 < d4; i4 += kDpThreads) dp_emit<T>(i4, src[i4], state_row, h_row, hi, lo, gamma);
  }
  if (hi && threadIdx.x == 0) a.next_ss[r] = s_sumsq;
}

void launch_dp_step(const DPStepArgs& a, int fp16, cudaStream_t s) {
  if (fp16)
    launch_ex(k_dp_step<__half>, dim3(a.hi - a.lo + 1), dim3(kDpThreads), 0, s, a);
  else
    launch_ex(k_dp_step<__nv_bfloat16>, dim3(a.hi - a.lo + 1), dim3(kDpThreads), 0, s, a);
}

// Backtrack from (L, n): back = 1 means layer i-1 (0-based) is skipped.
__global__ void k_dp_backtrack(const unsigned char* back, const float* val, int L, int n, int ncol,
                               unsigned char* mask, float* value) {
  griddep_launch();
  griddep_wait();
  int j = n;
  for (int i = L; i >= 1; --i) {
    const unsigned char b = back[(size_t)i * ncol + j];
    mask[i - 1] = b;
    if (b) --j;
  }
  *value = val[(size_t)L * ncol + n];
}

void launch_dp_backtrack(const unsigned char* back, const float* val, int L, int n, int ncol, unsigned char* mask,
                         float* value, cudaStream_t s) {
  launch_ex(k_dp_backtrack, dim3(1), dim3(1), 0, s, back, val, L, n, ncol, mask, value);
}

}  // namespace ssd
