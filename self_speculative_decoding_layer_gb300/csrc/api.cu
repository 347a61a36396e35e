// libssd host runtime: context, workspace layout, pass builders, CUDA-graph
// capture, the speculative decoding loop and the C ABI (include/ssd.h).
#include <cuda_runtime.h>
#include <math.h>
#include <stddef.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <string>
#include <vector>

#include "../../include/ssd.h"
#include "common.cuh"
#include "dytc.h"
#include "latency.h"
#include "kernels.h"
#include "misc.h"

using namespace ssd;

thread_local long long ssd::g_launches = 0;
thread_local bool ssd::g_pdl = true;

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
  size_t total = 0;
  size_t add(size_t bytes) {
    size_t off = total;
    total = align_up(total + bytes, 256);
    return off;
  }
};

struct Offsets {
  size_t st, desc, h, h2, q, o, act, logits, stash, am_part, am_cnt, acc_cnt, norm_ss, am1, am2, row_tok, drafts, tree_tok, parents, depth,
      anc, exp_node, exp_c0, exp_c1, prompt, out_tokens, dp_states, dp_val, dp_back, dp_mask, dp_value, sk_part, sk_cnt,
      trace, rope_cos,
      rope_sin, btab, kcache, vcache, mma_cnt, mma_xb, mma_xb_next, mma_scale, mma_ones, mma_part, total;
};

constexpr int kTraceSlots = 8192;
constexpr size_t kMmaPart = 24ull << 20;  // stream-K partial tiles of the tensor-core path

int n_pages_of(const ssd_model_config& c) { return (c.max_ctx + kPage - 1) / kPage; }

bool config_ok(const ssd_model_config* c) {
  if (!c) return false;
  if (c->n_layers < 1 || c->n_layers > kMaxLayers) return false;
  if (c->head_dim != 64 && c->head_dim != 128) return false;
  if (c->n_q_heads < 1 || c->n_kv_heads < 1 || c->n_q_heads % c->n_kv_heads) return false;
  if (c->d_model < 64 || c->d_model % 64 || c->ffn < 16 || c->ffn % 16) return false;
  if (c->vocab < 2 || c->vocab % 2) return false;
  if (c->dtype != SSD_BF16 && c->dtype != SSD_FP16) return false;
  if (c->max_rows < 1 || c->max_rows > kMaxRows) return false;
  if (c->max_ctx < c->max_rows + 1) return false;
  if ((c->n_q_heads * c->head_dim) % 8) return false;
  // the tcgen05 projection: at most 4096 weight tiles of 128 rows per matrix (the lm_head is the largest)
  if ((c->vocab + 127) / 128 > 4096) return false;
  return true;
}

Offsets layout_of(const ssd_model_config& c) {
  Layout L;
  Offsets o;
  const size_t R = c.max_rows, d = c.d_model, hq = (size_t)c.n_q_heads * c.head_dim;
  const size_t F = c.ffn, V = c.vocab;
  const int pages = n_pages_of(c);
  o.st = L.add(sizeof(DevState));
  o.desc = L.add(sizeof(PassDesc));
  o.h = L.add(R * d * 4);
  o.h2 = L.add(R * d * 4);  // the DP pass's pass rows alternate between h and h2
  o.q = L.add(R * hq * 4);
  o.o = L.add(R * hq * 4);
  o.act = L.add(R * F * 4);
  o.logits = L.add(R * V * 4);
  o.stash = L.add((size_t)(c.n_layers + 1) * R * d * 4);
  o.am_part = L.add(argmax_part_bytes((int)R));
  // RMSNorm hand-off: row sums of h^2 per output tile, or per tile and rank (up to 8) of the split-K kernel
  o.norm_ss = L.add(std::max<size_t>(d / 128, 1) * 8 * 64 * 4);
  o.am_cnt = L.add(R * 4);
  o.acc_cnt = L.add(4);  // rows whose argmax is done (fused acceptance)
  o.am1 = L.add(R * 4);
  o.am2 = L.add(R * 4);
  o.row_tok = L.add(R * 4);
  o.drafts = L.add(R * 4);
  o.tree_tok = L.add(R * 4);
  o.parents = L.add(R * 4);
  o.depth = L.add(R * 4);
  o.anc = L.add(R * 8);
  o.exp_node = L.add(R * 4);
  o.exp_c0 = L.add(R * 4);
  o.exp_c1 = L.add(R * 4);
  o.prompt = L.add((size_t)c.max_ctx * 4);
  o.out_tokens = L.add((size_t)c.max_ctx * 4);
  o.dp_states = L.add(2 * R * d * 4);
  o.dp_val = L.add((size_t)(c.n_layers + 1) * R * 4);
  o.dp_back = L.add((size_t)(c.n_layers + 1) * R);
  o.dp_mask = L.add(c.n_layers);
  o.dp_value = L.add(4);
  {
    // batch-1 GEMV merge: two partial sums per (unit, 1024-wide chunk), one counter per unit
    auto ch = [](size_t k) { return (k + 1023) / 1024; };
    const size_t nqkv = (size_t)(c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim / 2;
    const size_t nu = std::max<size_t>({nqkv, d / 2, F, V / 2});
    const size_t slots = std::max<size_t>({nqkv * ch(d), d / 2 * ch(hq), F * ch(d), d / 2 * ch(F), V / 2 * ch(d)});
    o.sk_part = L.add(slots * 2 * 4);
    o.sk_cnt = L.add(nu * 4);
  }
  o.trace = L.add((size_t)kTraceSlots * 3 * 8);
  o.rope_cos = L.add((size_t)c.max_ctx * (c.head_dim / 2) * 4);
  o.rope_sin = L.add((size_t)c.max_ctx * (c.head_dim / 2) * 4);
  o.btab = L.add((size_t)pages * 4);
  const size_t kv = (size_t)c.n_layers * pages * c.n_kv_heads * kPage * c.head_dim * 4;  // fp32 K and V
  o.kcache = L.add(kv);
  o.vcache = L.add(kv);
  o.mma_cnt = L.add(4096 * 4);
  {
    // tensor-core operand rows: [2][64][K] 16-bit for the widest input (preparation kernel / hand-off)
    const size_t kmax = std::max<size_t>({d, hq, F});
    o.mma_xb = L.add(2 * 64 * kmax * 2);
    o.mma_xb_next = L.add(2 * 64 * kmax * 2);
    o.mma_scale = L.add(64 * 4);
    o.mma_ones = L.add(64 * 4);
    o.mma_part = L.add(kMmaPart);
  }
  o.total = L.total;
  return o;
}

struct LayerW {
  const void *qkv, *o, *gu, *down, *g_attn, *g_ffn;
};

enum PassKind { PK_DRAFT = 0, PK_VERIFY = 1, PK_DP = 2, PK_AR = 3 };

struct Graph {
  cudaGraphExec_t exec = nullptr;
  long long kernels = 0;
  std::vector<int> trace_kind;
};

}  // namespace

struct ssd_ctx {
  ssd_model_config cfg;
  Offsets off;
  char* ws = nullptr;
  cudaStream_t stream = nullptr;
  cudaStream_t side = nullptr;  // captures the body graph of a conditional node
  int device = 0;
  int sms = 152;
  int fp16 = 0;
  bool weights = false;
  const void* embed = nullptr;
  const void* final_norm = nullptr;
  const void* lm_head = nullptr;
  std::vector<LayerW> layers;
  // host mirrors
  int t = 0;
  int pending = -1;
  int tgt_pos = -1;  // position of the CLaSp target token (host mirror)
  int last_dp_n = -1;  // n_skip of the last DP search (its table is in the workspace)
  bool have_target = false;
  bool have_pending = false;
  std::string err;
  int gemm_impl = 0;
  int use_graphs = 1;
  int use_pdl = 1;
  bool build_failed = false;  // a launcher refused its arguments while a pass was being enqueued
  bool in_graph = false;      // the pass being enqueued is captured into a graph of its own
  const int* gate = nullptr;  // while a draft step after the first is enqueued: its draft exit gate
  double beta[2][3] = {};         // latency model per activation mode (16-bit, int8), milliseconds
  bool have_beta[2] = {false, false};
  size_t pf_cap = 0;  // end-of-kernel L2 prefetch of the next weight matrix, bytes (0 = off)
  int tracing = 0;
  int trace_n = 0;
  std::vector<int> trace_kind;
  int timing = 0;
  int cycle_log = 0;
  std::vector<ssd_cycle_record> log;  // SSD_OPT_CYCLE_LOG
  std::map<std::string, Graph> graphs;
  std::vector<uint8_t> cur_skip;  // CLaSp mask in force
  // pinned staging
  int* h_pin = nullptr;
  size_t h_pin_n = 0;
  // timing
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> ev_pool;
  std::vector<std::pair<int, int>> ev_pending;  // (kind, pool index)
  double pass_ms[4] = {0, 0, 0, 0};
  int64_t pass_n[4] = {0, 0, 0, 0};
  size_t ev_next = 0;
  int64_t dp_runs = 0, ar_steps = 0, launches = 0, mma_fallbacks = 0;
  std::vector<double> ema;

  template <typename T = char>
  T* P(size_t o) const {
    return reinterpret_cast<T*>(ws + o);
  }
  DevState* st() const { return P<DevState>(off.st); }
  PassDesc* desc() const { return P<PassDesc>(off.desc); }
};

namespace {

ssd_status fail(ssd_ctx* c, ssd_status s, const std::string& msg) {
  if (c) c->err = msg;
  return s;
}

#define CU(call)                                                                           \
  do {                                                                                     \
    cudaError_t e_ = (call);                                                               \
    if (e_ != cudaSuccess) return fail(ctx, SSD_ERR_CUDA, std::string(#call ": ") + cudaGetErrorString(e_)); \
  } while (0)

// ---------------------------------------------------------------- launches

unsigned long long* trace_slot(ssd_ctx* ctx, int kind) {
  if (!ctx->tracing || ctx->trace_n >= kTraceSlots) return nullptr;
  ctx->trace_kind.push_back(kind);
  return ctx->P<unsigned long long>(ctx->off.trace) + (size_t)3 * ctx->trace_n++;
}

// Work distribution of the tensor-core projections: by shape, except in the test library, where
// SSD_OPT_GEMM_IMPL 4 forces split-K wherever the tiles fit and 5 forces stream-K.
int mma_mode(const ssd_ctx* ctx) {
#ifdef SSD_CROSSCHECK
  if (ctx->gemm_impl == 4) return 1;
  if (ctx->gemm_impl == 5) return 2;
#endif
  (void)ctx;
  return 0;
}

// Multi-row projections run on the tensor cores (everything but the test library's CUDA-core cross-check).
bool tc_rows(const ssd_ctx* ctx) { return ctx->gemm_impl == 0 || ctx->gemm_impl >= 4; }

void linear(ssd_ctx* ctx, LinearArgs a) {
  a.desc = ctx->desc();
  a.btab = ctx->P<int>(ctx->off.btab);
  a.n_pages = n_pages_of(ctx->cfg);
  a.n_q = ctx->cfg.n_q_heads;
  a.n_kv = ctx->cfg.n_kv_heads;
  a.hd = ctx->cfg.head_dim;
  a.rope_cos = ctx->P<float>(ctx->off.rope_cos);
  a.rope_sin = ctx->P<float>(ctx->off.rope_sin);
  a.kcache = ctx->P(ctx->off.kcache);
  a.vcache = ctx->P(ctx->off.vcache);
  a.eps = ctx->cfg.rms_eps;
  a.F = ctx->cfg.ffn;
  if (a.M > 1 && tc_rows(ctx) && !a.xb_ready) a.trace_prep = trace_slot(ctx, 20 + a.epi);
  a.trace = trace_slot(ctx, 10 + a.epi);
  a.sk_part = ctx->P<float>(ctx->off.sk_part);
  a.sk_cnt = ctx->P<int>(ctx->off.sk_cnt);
  a.err = &ctx->st()->err;
  a.gate = ctx->gate;
  a.mma_mode = mma_mode(ctx);
  if (a.pf_bytes > ctx->pf_cap) a.pf_bytes = ctx->pf_cap;
  if (!a.pf_bytes) a.pf = nullptr;
#ifdef SSD_CROSSCHECK
  // test library: the cross-check kernels selected by SSD_OPT_GEMM_IMPL
  if (ctx->gemm_impl == 1) {
    launch_linear_rows(a, ctx->fp16, ctx->stream);
    return;
  }
  if (a.M == 1 && ctx->gemm_impl == 2) {
    launch_gemv(a, ctx->fp16, ctx->stream);
    return;
  }
  if (a.M == 1 && ctx->gemm_impl == 3) {
    launch_gemv_bulk(a, ctx->fp16, ctx->sms, ctx->stream);
    return;
  }
#endif
  if (a.M == 1) {
    launch_gemv_rs(a, ctx->fp16, ctx->sms, ctx->stream);
    return;
  }
  MmaScratch sc{ctx->P(ctx->off.mma_xb), ctx->P<float>(ctx->off.mma_scale), ctx->P<float>(ctx->off.mma_ones),
                ctx->P<float>(ctx->off.mma_part), kMmaPart};
  if (!launch_mma(a, ctx->fp16, sc, ctx->P<int>(ctx->off.mma_cnt), ctx->sms, ctx->stream)) {
    // shapes are validated at ssd_create, so this is a tensor-map encoding failure: the pass is refused
    ctx->mma_fallbacks += 1;
    ctx->build_failed = true;
  }
}

// One-row passes (drafts, autoregressive steps, tree expansions) run their projections on the batch-1 GEMV,
// whose streaming loads land in L1: an SM's L1 is what its shared-memory carveout leaves, and an attention
// ring of 192 KB (six fp32 tiles, sized for a long context) leaves too little for the GEMVs that run on the
// SM after it (8B draft pass with 1636 cache slots: 12.30 ms with six slots, 9.74 ms with four; gate/up
// 51.3 -> 38.5 us).  Their ring is therefore capped at 128 KB; the tensor-core passes' projections stream
// by TMA and keep the whole ring.
constexpr int kBatch1RingBytes = 128 * 1024;

void attn_layout(ssd_ctx* ctx, int rows, AttnArgs& b) {
  const ssd_model_config& c = ctx->cfg;
  b.ring_cap = rows == 1 ? kBatch1RingBytes : 0;
  attention_layout(c.max_ctx + rows, rows, c.n_q_heads / c.n_kv_heads, c.n_kv_heads, 2, c.head_dim, b.ring_cap,
                   &b.qb, &b.n_split);
}

struct WRange {
  const void* p = nullptr;
  size_t bytes = 0;
  const void* gamma = nullptr;  // the RMSNorm gain applied to that matrix's input
};

size_t bytes_qkv(const ssd_model_config& c) { return (size_t)(c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim * c.d_model * 2; }

// The first weight matrix read after layer i when the layers in `skip` are bypassed:
// the next run layer's W_qkv, else the lm_head.
WRange next_weights(ssd_ctx* ctx, int i, const std::vector<uint8_t>* skip) {
  for (int j = i + 1; j < ctx->cfg.n_layers; ++j)
    if (!skip || !(*skip)[j]) return WRange{ctx->layers[j].qkv, bytes_qkv(ctx->cfg), ctx->layers[j].g_attn};
  return WRange{ctx->lm_head, (size_t)ctx->cfg.vocab * ctx->cfg.d_model * 2, ctx->final_norm};
}

bool norm_handoff_ok(ssd_ctx* ctx, int rows, bool int8) {
  return rows > 1 && !int8 && tc_rows(ctx) && ctx->cfg.d_model % 128 == 0;
}

// One transformer block (layer i) on `rows` pass rows held in h; `next` is
// the weight matrix the pass reads after this block (prefetched into L2).
// norm_in: the previous block's residual epilogue already wrote this block's
// normalised QKV operand rows; norm_out: write them for `next` (tensor-core
// rows only, see norm_handoff_ok).
// h_rows: the pass rows (default: the h buffer); qkv_ss: slots of the RMSNorm hand-off the QKV projection reads
// (default: what the previous block's down projection wrote; the DP step writes one per row).
void layer(ssd_ctx* ctx, int i, int rows, bool int8, float* stash_next, WRange next, bool norm_in = false,
           bool norm_out = false, float* h_rows = nullptr, int qkv_ss = 0) {
  const ssd_model_config& c = ctx->cfg;
  const LayerW& w = ctx->layers[i];
  float* h = h_rows ? h_rows : ctx->P<float>(ctx->off.h);
  float* q = ctx->P<float>(ctx->off.q);
  float* o = ctx->P<float>(ctx->off.o);
  float* act = ctx->P<float>(ctx->off.act);
  const int hq = c.n_q_heads * c.head_dim;
  // tensor-core rows without int8: attention and the SwiGLU epilogue write the O and down projections'
  // 16-bit operand rows themselves, so those two projections need no preparation kernel
  void* handoff = (rows > 1 && !int8 && tc_rows(ctx)) ? ctx->P(ctx->off.mma_xb_next) : nullptr;
  const bool norm = norm_handoff_ok(ctx, rows, int8);
  void* xbn = ctx->P(ctx->off.mma_xb);
  float* ss = ctx->P<float>(ctx->off.norm_ss);
  // slots the hand-off producers write: the down projection (K = ffn) for the next block's QKV, W_o for gate/up
  const int ss_after_down = mma_ss_slots(c.d_model, c.ffn, rows, ctx->fp16, ctx->sms, mma_mode(ctx));
  const int ss_after_o = mma_ss_slots(c.d_model, hq, rows, ctx->fp16, ctx->sms, mma_mode(ctx));
  LinearArgs a{};
  a.W = w.qkv;
  a.N = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
  a.K = c.d_model;
  a.X = h;
  a.ldx = c.d_model;
  a.M = rows;
  a.gamma = w.g_attn;
  a.int8 = int8;
  a.epi = EPI_QKV;
  a.out = q;
  a.ldo = hq;
  a.layer = i;
  if (norm && norm_in) {
    a.xb_ready = xbn;
    a.ss_in = ss;
    a.ss_tiles = qkv_ss ? qkv_ss : ss_after_down;
  }
  a.pf = w.o;
  a.pf_bytes = (size_t)c.d_model * hq * 2;
  linear(ctx, a);

  AttnArgs b{};
  b.desc = ctx->desc();
  b.q = q;
  b.kcache = ctx->P(ctx->off.kcache);
  b.vcache = ctx->P(ctx->off.vcache);
  b.btab = ctx->P<int>(ctx->off.btab);
  b.n_pages = n_pages_of(c);
  b.layer = i;
  b.n_q = c.n_q_heads;
  b.n_kv = c.n_kv_heads;
  b.hd = c.head_dim;
  b.max_keys = ctx->cfg.max_ctx + rows;
  b.err = &ctx->st()->err;
  b.out = o;
  b.rows = rows;
  attn_layout(ctx, rows, b);
  b.pf = w.gu;
  b.pf_bytes = std::min(ctx->pf_cap, (size_t)2 * c.ffn * c.d_model * 2);
  if (!b.pf_bytes) b.pf = nullptr;
  b.trace = trace_slot(ctx, 2);
  b.gate = ctx->gate;
  // a pass replayed as its own graph starts after the previous one has completed and writes no slot below
  // the committed length before its attention: those prefix tiles may be copied before the dependency wait
  b.committed = &ctx->st()->t;
  b.early = ctx->in_graph ? 1 : 0;
  // the first stages of every gate/up row into L2 during attention, 16 MB in all (in 256-byte steps, two
  // 64-wide K stages), when the gate/up projection runs one tile pair per CTA from column 0: 8B 7-row
  // verify 3.251 -> 3.220 ms, DP 3.596 -> 3.582 ms on one box; with 32 MB on the 70B shape, whose gate/up
  // runs stream-K (CTAs starting mid-tile), the verify went 26.34 -> 26.52 ms
  if (rows > 1 && !int8 && tc_rows(ctx) &&
      mma_split_ways(c.ffn, c.d_model, rows, 2, ctx->fp16, ctx->sms, mma_mode(ctx)) == 1) {
    const long long head = std::min<long long>((16LL << 20) / (2LL * c.ffn) / 256 * 256, 2LL * c.d_model);
    if (head > 0) {
      b.head_pf = reinterpret_cast<const char*>(w.gu);
      b.head_rows = 2 * c.ffn;
      b.head_stride = 2 * c.d_model;
      b.head_bytes = (int)head;
    }
  }
  b.xb_next = handoff;
  b.next_mp = mma_rows_pad(rows);
  b.xb_fp16 = ctx->fp16;
  if (!launch_attention(b, 2, ctx->stream)) ctx->build_failed = true;

  LinearArgs e{};
  e.W = w.o;
  e.N = c.d_model;
  e.K = hq;
  e.X = o;
  e.ldx = hq;
  e.M = rows;
  e.int8 = int8;
  e.epi = EPI_RESID;
  e.out = h;
  e.ldo = c.d_model;
  e.layer = i;
  e.xb_ready = handoff;
  if (norm) {  // gate/up's normalised operand rows
    e.xbn_out = xbn;
    e.gamma_next = w.g_ffn;
    e.ss_out = ss;
    e.next_mp = mma_rows_pad(rows);
  }
  e.pf = w.gu;
  e.pf_bytes = (size_t)2 * c.ffn * c.d_model * 2;
  linear(ctx, e);

  LinearArgs f{};
  f.W = w.gu;
  f.N = 2 * c.ffn;
  f.K = c.d_model;
  f.X = h;
  f.ldx = c.d_model;
  f.M = rows;
  f.gamma = w.g_ffn;
  f.int8 = int8;
  f.epi = EPI_SWIGLU;
  f.out = act;
  f.ldo = c.ffn;
  f.layer = i;
  f.xb_next = handoff;
  f.next_mp = mma_rows_pad(rows);
  if (norm) {
    f.xb_ready = xbn;
    f.ss_in = ss;
    f.ss_tiles = ss_after_o;
  }
  f.pf = w.down;
  f.pf_bytes = (size_t)c.ffn * c.d_model * 2;
  linear(ctx, f);

  LinearArgs g{};
  g.W = w.down;
  g.N = c.d_model;
  g.K = c.ffn;
  g.X = act;
  g.ldx = c.ffn;
  g.M = rows;
  g.int8 = int8;
  g.epi = EPI_RESID;
  g.out = h;
  g.ldo = c.d_model;
  g.stash = stash_next;
  g.layer = i;
  g.xb_ready = handoff;
  if (norm && norm_out) {  // the next block's (or lm_head's) normalised operand rows
    g.xbn_out = xbn;
    g.gamma_next = next.gamma;
    g.ss_out = ss;
    g.next_mp = mma_rows_pad(rows);
  }
  g.pf = next.p;
  g.pf_bytes = next.bytes;
  linear(ctx, g);
}

float* stash_layer(ssd_ctx* ctx, int l) {
  return ctx->P<float>(ctx->off.stash) + (size_t)l * ctx->cfg.max_rows * ctx->cfg.d_model;
}

// Final RMSNorm + lm_head over `rows` rows starting at pass row `row0`,
// logits into rows 0.. of the logits buffer, then greedy argmax / top-2.
void lm_head(ssd_ctx* ctx, int row0, int rows, int* out1, int* out2, WRange next = WRange{}, bool norm_in = false,
             ArgmaxExit ex = ArgmaxExit{}, AcceptArgs acc = AcceptArgs{}) {
  const ssd_model_config& c = ctx->cfg;
  LinearArgs a{};
  a.W = ctx->lm_head;
  a.N = c.vocab;
  a.K = c.d_model;
  a.X = ctx->P<float>(ctx->off.h) + (size_t)row0 * c.d_model;
  a.ldx = c.d_model;
  a.M = rows;
  a.row0 = row0;
  a.gamma = ctx->final_norm;
  a.epi = EPI_LOGITS;
  a.out = ctx->P<float>(ctx->off.logits);
  a.ldo = c.vocab;
  a.pf = next.p;
  a.pf_bytes = next.bytes;
  if (norm_in && row0 == 0 && norm_handoff_ok(ctx, rows, false)) {
    a.xb_ready = ctx->P(ctx->off.mma_xb);
    a.ss_in = ctx->P<float>(ctx->off.norm_ss);
    a.ss_tiles = mma_ss_slots(c.d_model, c.ffn, rows, ctx->fp16, ctx->sms, mma_mode(ctx));  // the last down projection's
  }
  linear(ctx, a);
  launch_argmax(ctx->P<float>(ctx->off.logits), rows, c.vocab, c.vocab, out1, out2, ctx->P(ctx->off.am_part),
                ctx->P<int>(ctx->off.am_cnt), ctx->stream, ex, acc);
}

BeginArgs begin_base(ssd_ctx* ctx, int kind, int rows) {
  BeginArgs b{};
  b.kind = kind;
  b.rows = rows;
  b.st = ctx->st();
  b.desc = ctx->desc();
  b.E = ctx->embed;
  b.d = ctx->cfg.d_model;
  b.vocab = ctx->cfg.vocab;
  b.h = ctx->P<float>(ctx->off.h);
  b.ldh = ctx->cfg.d_model;
  b.row_tok = ctx->P<int>(ctx->off.row_tok);
  b.trace = trace_slot(ctx, 0);
  return b;
}

// ---- pass builders (each enqueues one pass on ctx->stream)

void pass_prefill_chunk(ssd_ctx* ctx, int off, int n, bool last) {
  BeginArgs b = begin_base(ctx, BEGIN_CAUSAL, n);
  b.tok = ctx->P<int>(ctx->off.prompt);
  b.tok_offset = off;
  b.first_pending = 0;
  b.stash0 = stash_layer(ctx, 0);
  launch_begin(b, ctx->fp16, ctx->stream);
  for (int i = 0; i < ctx->cfg.n_layers; ++i)
    layer(ctx, i, n, false, stash_layer(ctx, i + 1), next_weights(ctx, i, nullptr), i > 0, i + 1 < ctx->cfg.n_layers);
  int* am1 = ctx->P<int>(ctx->off.am1);
  if (last) lm_head(ctx, n - 1, 1, am1, ctx->P<int>(ctx->off.am2));
  launch_advance(ctx->st(), n, am1, last ? 1 : 0, nullptr, ctx->stream);
}

void pass_ar(ssd_ctx* ctx, int* out_tokens) {
  BeginArgs b = begin_base(ctx, BEGIN_CAUSAL, 1);
  b.first_pending = 1;
  b.tok = ctx->P<int>(ctx->off.drafts);
  b.stash0 = stash_layer(ctx, 0);
  launch_begin(b, ctx->fp16, ctx->stream);
  for (int i = 0; i < ctx->cfg.n_layers; ++i) layer(ctx, i, 1, false, stash_layer(ctx, i + 1), next_weights(ctx, i, nullptr));
  int* am1 = ctx->P<int>(ctx->off.am1);
  lm_head(ctx, 0, 1, am1, ctx->P<int>(ctx->off.am2), next_weights(ctx, -1, nullptr));
  launch_advance(ctx->st(), 1, am1, 1, out_tokens, ctx->stream);
}

void draft_forward(ssd_ctx* ctx, int step, const std::vector<uint8_t>& skip, bool int8, ArgmaxExit ex, int exit_k) {
  int* drafts = ctx->P<int>(ctx->off.drafts);
  BeginArgs b = begin_base(ctx, BEGIN_DRAFT, 1);
  b.step = step;
  b.tok = drafts;
  b.row_tok = nullptr;
  b.exit_k = exit_k;
  launch_begin(b, ctx->fp16, ctx->stream);
  for (int i = 0; i < ctx->cfg.n_layers; ++i)
    if (!skip[i]) layer(ctx, i, 1, int8, nullptr, next_weights(ctx, i, &skip));
  lm_head(ctx, 0, 1, ex.dyn ? drafts : drafts + step, nullptr, next_weights(ctx, -1, &skip), false, ex);
}

// Draft exit inside a captured graph: a conditional WHILE node runs one draft forward per iteration
// (the step is DevState::draft_n) and each iteration's argmax sets the loop condition, so the forwards
// after an exit are never launched.  The body is captured on the side stream into the node's graph.
// False if a graph call failed (the pass is then not usable).
bool pass_draft_loop(ssd_ctx* ctx, int k, const std::vector<uint8_t>& skip, bool int8, float exit_thr) {
  launch_draft_reset(ctx->st(), ctx->P<int>(ctx->off.drafts), k, ctx->stream);
  cudaStreamCaptureStatus cs;
  cudaGraph_t g = nullptr;
  const cudaGraphNode_t* deps = nullptr;
  const cudaGraphEdgeData* edges = nullptr;
  size_t nd = 0;
  if (cudaStreamGetCaptureInfo(ctx->stream, &cs, nullptr, &g, &deps, &edges, &nd) != cudaSuccess ||
      cs != cudaStreamCaptureStatusActive)
    return false;
  cudaGraphConditionalHandle h;
  if (cudaGraphConditionalHandleCreate(&h, g, 1u, cudaGraphCondAssignDefault) != cudaSuccess) return false;
  cudaGraphNodeParams np = {};
  np.type = cudaGraphNodeTypeConditional;
  np.conditional.handle = h;
  np.conditional.type = cudaGraphCondTypeWhile;
  np.conditional.size = 1;
  cudaGraphNode_t node;
  if (cudaGraphAddNode(&node, g, deps, nullptr, nd, &np) != cudaSuccess) return false;
  if (cudaStreamUpdateCaptureDependencies(ctx->stream, &node, nullptr, 1, cudaStreamSetCaptureDependencies) !=
      cudaSuccess)
    return false;
  cudaGraph_t body = np.conditional.phGraph_out[0];
  if (cudaStreamBeginCaptureToGraph(ctx->side, body, nullptr, nullptr, 0, cudaStreamCaptureModeRelaxed) !=
      cudaSuccess)
    return false;
  cudaStream_t main = ctx->stream;
  ctx->stream = ctx->side;
  ArgmaxExit ex{ctx->st(), exit_thr, 0, 1, k, 1, h};
  draft_forward(ctx, -1, skip, int8, ex, 0);
  ctx->stream = main;
  cudaGraph_t out = nullptr;
  return cudaStreamEndCapture(ctx->side, &out) == cudaSuccess;
}

// K draft forwards.  With a draft exit threshold (exit_thr > 0) every step's argmax also
// computes the draft's top-1 probability and closes the gate when it is below the
// threshold; the kernels of the later steps then return right after their dependency
// wait, so the pass keeps its fixed shape (one graph) and the drafts not reached stay -1.
void pass_draft(ssd_ctx* ctx, int k, const std::vector<uint8_t>& skip, bool int8, float exit_thr) {
  const bool exit_on = exit_thr > 0.f;
  if (exit_on && ctx->use_graphs && !ctx->tracing && k > 1) {
    if (!pass_draft_loop(ctx, k, skip, int8, exit_thr)) ctx->build_failed = true;
    return;
  }
  for (int s = 0; s < k; ++s) {
    ctx->gate = (exit_on && s > 0) ? &ctx->st()->draft_live : nullptr;
    ArgmaxExit ex{};
    if (exit_on) ex = ArgmaxExit{ctx->st(), exit_thr, s};
    draft_forward(ctx, s, skip, int8, ex, exit_on ? k : 0);
  }
  ctx->gate = nullptr;
}

void pass_verify(ssd_ctx* ctx, int n_rows, bool tree, int* out_tokens) {
  BeginArgs b = begin_base(ctx, tree ? BEGIN_TREE : BEGIN_CAUSAL, n_rows);
  if (tree) {
    b.tok = ctx->P<int>(ctx->off.tree_tok);
    b.depth = ctx->P<int>(ctx->off.depth);
    b.anc = ctx->P<unsigned long long>(ctx->off.anc);
  } else {
    b.tok = ctx->P<int>(ctx->off.drafts);
    b.first_pending = 1;
  }
  b.stash0 = stash_layer(ctx, 0);
  launch_begin(b, ctx->fp16, ctx->stream);
  for (int i = 0; i < ctx->cfg.n_layers; ++i)
    layer(ctx, i, n_rows, false, stash_layer(ctx, i + 1), next_weights(ctx, i, nullptr), i > 0, true);
  int* am1 = ctx->P<int>(ctx->off.am1);
  // greedy acceptance and rollback run in the argmax launch's last CTA
  const AcceptArgs acc{ctx->st(), ctx->P<int>(ctx->off.row_tok), tree ? ctx->P<int>(ctx->off.parents) : nullptr, n_rows,
                       out_tokens, ctx->P<int>(ctx->off.acc_cnt)};
  lm_head(ctx, 0, n_rows, am1, ctx->P<int>(ctx->off.am2), WRange{}, true, ArgmaxExit{}, acc);
  if (tree)
    launch_compact(ctx->st(), ctx->P(ctx->off.kcache), ctx->P(ctx->off.vcache), ctx->P<int>(ctx->off.btab),
                   n_pages_of(ctx->cfg), ctx->cfg.n_layers, ctx->cfg.n_kv_heads, ctx->cfg.head_dim, ctx->fp16,
                   ctx->stream);
}

// Vertical cascade: the higher draft level runs the pending token and the k lower-level drafts as one
// multi-row pass over its layers (KV to scratch slots t..t+k), then keeps the drafts it agrees with.
void pass_draft_verify(ssd_ctx* ctx, int k, const std::vector<uint8_t>& skip, bool int8) {
  const int rows = k + 1;
  BeginArgs b = begin_base(ctx, BEGIN_CAUSAL, rows);
  b.tok = ctx->P<int>(ctx->off.drafts);
  b.first_pending = 1;
  b.row_tok = nullptr;
  launch_begin(b, ctx->fp16, ctx->stream);
  bool first = true;
  for (int i = 0; i < ctx->cfg.n_layers; ++i) {
    if (skip[i]) continue;
    layer(ctx, i, rows, int8, nullptr, next_weights(ctx, i, &skip), !first, true);
    first = false;
  }
  int* am1 = ctx->P<int>(ctx->off.am1);
  lm_head(ctx, 0, rows, am1, nullptr, WRange{}, !first && norm_handoff_ok(ctx, rows, int8));
  launch_draft_accept(am1, ctx->P<int>(ctx->off.drafts), k, ctx->stream);
}

void pass_expand(ssd_ctx* ctx, const std::vector<uint8_t>& skip, bool int8) {
  BeginArgs b = begin_base(ctx, BEGIN_EXPAND, 1);
  b.tok = ctx->P<int>(ctx->off.tree_tok);
  b.depth = ctx->P<int>(ctx->off.depth);
  b.anc = ctx->P<unsigned long long>(ctx->off.anc);
  b.exp_node = ctx->P<int>(ctx->off.exp_node);
  b.row_tok = nullptr;
  launch_begin(b, ctx->fp16, ctx->stream);
  for (int i = 0; i < ctx->cfg.n_layers; ++i)
    if (!skip[i]) layer(ctx, i, 1, int8, nullptr, next_weights(ctx, i, &skip));
  int* am1 = ctx->P<int>(ctx->off.am1);
  int* am2 = ctx->P<int>(ctx->off.am2);
  lm_head(ctx, 0, 1, am1, am2);
  launch_store_children(ctx->st(), ctx->P<int>(ctx->off.tree_tok), ctx->P<int>(ctx->off.exp_c0),
                        ctx->P<int>(ctx->off.exp_c1), am1, am2, ctx->stream);
}

void dp_range(int L, int n, int i, int& lo, int& hi) {
  lo = std::max(0, n - (L - i));
  hi = std::min(i, n);
}

void pass_dp(ssd_ctx* ctx, int n) {
  const ssd_model_config& c = ctx->cfg;
  const int L = c.n_layers, d = c.d_model, ncol = c.max_rows;
  float* states[2] = {ctx->P<float>(ctx->off.dp_states), ctx->P<float>(ctx->off.dp_states) + (size_t)ncol * d};
  float* hbuf[2] = {ctx->P<float>(ctx->off.h), ctx->P<float>(ctx->off.h2)};
  float* val = ctx->P<float>(ctx->off.dp_val);
  unsigned char* back = ctx->P<unsigned char>(ctx->off.dp_back);
  void* xb = ctx->P(ctx->off.mma_xb);
  float* ss = ctx->P<float>(ctx->off.norm_ss);
  // one descriptor for every layer: row r at the target's position, in scratch slot t + r, seeing the
  // committed prefix before the target and its own K/V (launch row counts come from the launches)
  BeginArgs b = begin_base(ctx, BEGIN_DP, n + 1);
  b.row_tok = nullptr;
  launch_begin(b, ctx->fp16, ctx->stream);
  // the rows of layer 0: state(0, 0) alone
  launch_dp_init(ctx->st(), stash_layer(ctx, 0), d, states[0], val, back, hbuf[0], nullptr, nullptr, nullptr, 0,
                 ctx->fp16, ctx->stream);
  for (int i = 1; i <= L; ++i) {
    int lo_p, hi_p, lo, hi;
    dp_range(L, n, i - 1, lo_p, hi_p);
    dp_range(L, n, i, lo, hi);
    const int rows = hi_p - lo_p + 1;  // states (i-1, lo_p..hi_p) run through layer i-1
    float* h = hbuf[(i - 1) & 1];
    // their QKV operand rows were handed over by the previous DP step when this is a tensor-core layer
    layer(ctx, i - 1, rows, false, nullptr, next_weights(ctx, i - 1, nullptr), norm_handoff_ok(ctx, rows, false),
          false, h, 1);
    DPStepArgs s{};
    s.st = ctx->st();
    s.i = i;
    s.lo = lo;
    s.hi = hi;
    s.lo_prev = lo_p;
    s.hi_prev = hi_p;
    s.h = h;
    s.ldh = d;
    s.states_old = states[(i - 1) & 1];
    s.states_new = states[i & 1];
    s.stash_i = stash_layer(ctx, i);
    s.d = d;
    s.val = val;
    s.back = back;
    s.ncol = ncol;
    if (i < L) {  // the next layer's pass rows: states (i, lo..hi)
      const int next_rows = hi - lo + 1;
      s.next_h = hbuf[i & 1];
      if (norm_handoff_ok(ctx, next_rows, false)) {
        s.next_xb = xb;
        s.next_ss = ss;
        s.next_gamma = ctx->layers[i].g_attn;
        s.next_mp = mma_rows_pad(next_rows);
      }
    }
    launch_dp_step(s, ctx->fp16, ctx->stream);
  }
  launch_dp_backtrack(back, val, L, n, ncol, ctx->P<unsigned char>(ctx->off.dp_mask),
                      ctx->P<float>(ctx->off.dp_value), ctx->stream);
}

// ---------------------------------------------------------------- graphs

std::string mask_key(const std::vector<uint8_t>& m) {
  std::string s;
  for (uint8_t b : m) s.push_back(b ? '1' : '0');
  return s;
}

template <typename F>
ssd_status run_pass(ssd_ctx* ctx, const std::string& key0, F&& build) {
  g_pdl = ctx->use_pdl != 0;
  const std::string key = ctx->tracing ? key0 + "/trace" : key0;
  if (ctx->tracing) {
    ctx->trace_n = 0;
    ctx->trace_kind.clear();
    CU(cudaMemsetAsync(ctx->P(ctx->off.trace), 0, (size_t)kTraceSlots * 3 * 8, ctx->stream));
  }
  ctx->build_failed = false;
  if (!ctx->use_graphs) {
    const long long before = g_launches;
    build();
    ctx->launches += g_launches - before;
    CU(cudaGetLastError());
    if (ctx->build_failed) return fail(ctx, SSD_ERR_CUDA, "a kernel launch was refused while enqueueing the pass");
    return SSD_OK;
  }
  auto it = ctx->graphs.find(key);
  if (it == ctx->graphs.end()) {
    if (ctx->graphs.size() > 64) {
      for (auto& g : ctx->graphs) cudaGraphExecDestroy(g.second.exec);
      ctx->graphs.clear();
    }
    cudaGraph_t g;
    CU(cudaStreamBeginCapture(ctx->stream, cudaStreamCaptureModeRelaxed));
    const long long before = g_launches;
    ctx->in_graph = true;
    build();
    ctx->in_graph = false;
    const long long n_kernels = g_launches - before;
    cudaError_t e = cudaStreamEndCapture(ctx->stream, &g);
    if (e != cudaSuccess) return fail(ctx, SSD_ERR_CUDA, std::string("capture: ") + cudaGetErrorString(e));
    if (ctx->build_failed) {
      cudaGraphDestroy(g);
      return fail(ctx, SSD_ERR_CUDA, "a kernel launch was refused while capturing the pass");
    }
    Graph gr;
    gr.kernels = n_kernels;
    gr.trace_kind = ctx->trace_kind;
    e = cudaGraphInstantiate(&gr.exec, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) return fail(ctx, SSD_ERR_CUDA, std::string("instantiate: ") + cudaGetErrorString(e));
    it = ctx->graphs.emplace(key, gr).first;
  }
  CU(cudaGraphLaunch(it->second.exec, ctx->stream));
  ctx->launches += it->second.kernels;
  if (ctx->tracing) {
    ctx->trace_kind = it->second.trace_kind;
    ctx->trace_n = (int)ctx->trace_kind.size();
  }
  return SSD_OK;
}

void drop_graphs(ssd_ctx* ctx) {
  for (auto& g : ctx->graphs) cudaGraphExecDestroy(g.second.exec);
  ctx->graphs.clear();
}

// timing helpers: events around passes (outside the graphs)
int timer_begin(ssd_ctx* ctx) {
  if (!ctx->timing) return -1;
  if (ctx->ev_next >= ctx->ev_pool.size()) {
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    ctx->ev_pool.push_back({a, b});
  }
  int idx = (int)ctx->ev_next++;
  cudaEventRecord(ctx->ev_pool[idx].first, ctx->stream);
  return idx;
}

void timer_end(ssd_ctx* ctx, int idx, int kind) {
  if (idx < 0) return;
  cudaEventRecord(ctx->ev_pool[idx].second, ctx->stream);
  ctx->ev_pending.push_back({kind, idx});
}

void timer_collect(ssd_ctx* ctx) {
  for (auto& p : ctx->ev_pending) {
    float ms = 0.f;
    cudaEventElapsedTime(&ms, ctx->ev_pool[p.second].first, ctx->ev_pool[p.second].second);
    ctx->pass_ms[p.first] += ms;
    ctx->pass_n[p.first] += 1;
  }
  ctx->ev_pending.clear();
  ctx->ev_next = 0;
}

ssd_status sync(ssd_ctx* ctx) {
  CU(cudaStreamSynchronize(ctx->stream));
  timer_collect(ctx);
  return SSD_OK;
}

ssd_status h2d(ssd_ctx* ctx, void* dst, const void* src, size_t bytes) {
  CU(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, ctx->stream));
  return SSD_OK;
}

ssd_status d2h(ssd_ctx* ctx, void* dst, const void* src, size_t bytes) {
  CU(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, ctx->stream));
  return SSD_OK;
}

#define TRY(x)                      \
  do {                              \
    ssd_status s_ = (x);            \
    if (s_ != SSD_OK) return s_;    \
  } while (0)

ssd_status read_state(ssd_ctx* ctx, DevState* out) {
  TRY(d2h(ctx, out, ctx->st(), sizeof(DevState)));
  TRY(sync(ctx));
  ctx->t = out->t;
  ctx->pending = out->pending;
  ctx->tgt_pos = out->tgt_pos;
  if (out->err == kDevErrToken)
    return fail(ctx, SSD_ERR_CUDA, "a token id outside the vocabulary reached the embedding");
  if (out->err) return fail(ctx, SSD_ERR_TIMEOUT, "a bounded device-side wait gave up");
  return SSD_OK;
}

// upload helper through the pinned staging buffer (synchronous w.r.t. the host buffer)
ssd_status upload(ssd_ctx* ctx, void* dst, const void* src, size_t bytes) {
  if (bytes == 0) return SSD_OK;
  TRY(sync(ctx));  // the staging buffer may still be read by an earlier copy
  if (bytes > ctx->h_pin_n) return fail(ctx, SSD_ERR_CAPACITY, "staging buffer too small");
  memcpy(ctx->h_pin, src, bytes);
  return h2d(ctx, dst, ctx->h_pin, bytes);
}

ssd_status set_dev_int(ssd_ctx* ctx, int* dst, int v) { return upload(ctx, dst, &v, sizeof(int)); }

bool need_state(ssd_ctx* ctx) { return ctx->weights && ctx->have_pending; }

ssd_status check_skip(ssd_ctx* ctx, const uint8_t* m) {
  if (!m) return fail(ctx, SSD_ERR_INVALID_ARG, "skip mask is null");
  return SSD_OK;
}

// Layers a draft does not run: its skip set plus the last `early_exit` layers (an early exit after
// layer L - e - 1 is the same forward as bypassing the last e layers).
void add_early_exit(std::vector<uint8_t>& mask, int e) {
  for (int i = (int)mask.size() - e; i < (int)mask.size(); ++i)
    if (i >= 0) mask[i] = 1;
}

std::vector<uint8_t> level_mask(const ssd_model_config& c, const ssd_policy* p, int l) {
  std::vector<uint8_t> m(p->level_skip + (size_t)l * c.n_layers, p->level_skip + (size_t)(l + 1) * c.n_layers);
  for (auto& b : m) b = b ? 1 : 0;
  if (p->level_exit) add_early_exit(m, p->level_exit[l]);
  return m;
}

std::vector<double> level_costs(const ssd_model_config& c, const ssd_policy* p) {
  const int64_t hd = c.head_dim, d = c.d_model, F = c.ffn;
  const int64_t qkv = (int64_t)(c.n_q_heads + 2 * c.n_kv_heads) * hd;
  const int64_t w_layer = 2 * (qkv * d + d * c.n_q_heads * hd + 2 * F * d + d * F);
  const int64_t w_lm = 2 * (int64_t)c.vocab * d;
  const int64_t full = (int64_t)c.n_layers * w_layer + w_lm;
  std::vector<double> out;
  for (int l = 0; l < p->n_levels; ++l) {
    int64_t skipped = 0;
    for (uint8_t b : level_mask(c, p, l)) skipped += b;
    const int64_t num = (c.n_layers - skipped) * w_layer + w_lm;
    out.push_back((double)num / (double)full);
  }
  return out;
}

ssd_status validate_tree(ssd_ctx* ctx, const int32_t* parents, int n) {
  if (parents[0] != -1) return fail(ctx, SSD_ERR_INVALID_ARG, "tree_parents[0] must be -1");
  for (int c = 1; c < n; ++c)
    if (parents[c] < 0 || parents[c] >= c) return fail(ctx, SSD_ERR_INVALID_ARG, "tree_parents[c] must be in [0, c)");
  return SSD_OK;
}

// Upload a tree (tokens[1..], parents, depth, ancestor masks) for a tree verify.
ssd_status upload_tree(ssd_ctx* ctx, const int32_t* tokens, const int32_t* parents, int n) {
  std::vector<int> buf(4 * kMaxRows, 0);
  std::vector<unsigned long long> anc(n, 0);
  int* tok = buf.data();
  int* par = buf.data() + kMaxRows;
  int* dep = buf.data() + 2 * kMaxRows;
  for (int c = 0; c < n; ++c) {
    tok[c] = tokens ? tokens[c] : 0;
    par[c] = parents[c];
    dep[c] = c == 0 ? 0 : dep[parents[c]] + 1;
    anc[c] = (c == 0 ? 0ull : anc[parents[c]]) | (1ull << c);
  }
  if (tokens) TRY(upload(ctx, ctx->P(ctx->off.tree_tok), tok, n * 4));
  TRY(upload(ctx, ctx->P(ctx->off.parents), par, n * 4));
  TRY(upload(ctx, ctx->P(ctx->off.depth), dep, n * 4));
  TRY(upload(ctx, ctx->P(ctx->off.anc), anc.data(), n * 8));
  return SSD_OK;
}

// Per-cycle log entry for the verify pass that just ran (rows verify rows; tree: the plan's parents, else a
// chain); s is the device state read after it.  Reads the rows' tokens and argmax (a synchronising copy).
ssd_status log_cycle(ssd_ctx* ctx, int kind, int t_before, int rows, const std::vector<int>* parents,
                     const DevState& s) {
  ssd_cycle_record r;
  memset(&r, 0, sizeof(r));
  r.kind = kind;
  r.t = t_before;
  r.n_rows = rows;
  r.n_acc = s.n_acc;
  r.bonus = s.bonus;
  TRY(d2h(ctx, r.tokens, ctx->P(ctx->off.row_tok), (size_t)rows * 4));
  TRY(d2h(ctx, r.argmax, ctx->P(ctx->off.am1), (size_t)rows * 4));
  TRY(sync(ctx));
  for (int c = 0; c < rows; ++c) r.parents[c] = parents ? (*parents)[c] : c - 1;
  for (int i = 0; i <= s.n_acc && i <= kMaxRows; ++i) r.path[i] = s.path[i];
  for (size_t l = 0; l < ctx->ema.size() && l < 3; ++l) r.ema[l] = ctx->ema[l];
  ctx->log.push_back(r);
  return SSD_OK;
}

ssd_status launch_ar(ssd_ctx* ctx, int* out) {
  int ti = timer_begin(ctx);
  TRY(run_pass(ctx, "ar", [&] { pass_ar(ctx, out); }));
  timer_end(ctx, ti, PK_AR);
  return SSD_OK;
}

ssd_status launch_draft(ssd_ctx* ctx, const std::vector<uint8_t>& skip, int int8, int k, float exit_thr = 0.f) {
  int ti = timer_begin(ctx);
  char thr[32];
  snprintf(thr, sizeof(thr), "%a", exit_thr > 0.f ? exit_thr : 0.f);
  TRY(run_pass(ctx, "draft/" + mask_key(skip) + "/" + std::to_string(int8) + "/" + std::to_string(k) + "/" + thr,
               [&] { pass_draft(ctx, k, skip, int8 != 0, exit_thr); }));
  timer_end(ctx, ti, PK_DRAFT);
  return SSD_OK;
}

ssd_status launch_verify(ssd_ctx* ctx, int rows, bool tree, int* out) {
  int ti = timer_begin(ctx);
  TRY(run_pass(ctx, std::string(tree ? "tree/" : "verify/") + std::to_string(rows) + (out ? "/o" : ""),
               [&] { pass_verify(ctx, rows, tree, out); }));
  timer_end(ctx, ti, PK_VERIFY);
  return SSD_OK;
}

ssd_status launch_dp(ssd_ctx* ctx, int n) {
  int ti = timer_begin(ctx);
  TRY(run_pass(ctx, "dp/" + std::to_string(n), [&] { pass_dp(ctx, n); }));
  timer_end(ctx, ti, PK_DP);
  ctx->dp_runs += 1;
  return SSD_OK;
}

ssd_status launch_draft_verify(ssd_ctx* ctx, const std::vector<uint8_t>& skip, int int8, int k) {
  int ti = timer_begin(ctx);
  TRY(run_pass(ctx, "dverify/" + mask_key(skip) + "/" + std::to_string(int8) + "/" + std::to_string(k),
               [&] { pass_draft_verify(ctx, k, skip, int8 != 0); }));
  timer_end(ctx, ti, PK_DRAFT);
  return SSD_OK;
}

ssd_status launch_expand(ssd_ctx* ctx, const std::vector<uint8_t>& skip, int int8) {
  int ti = timer_begin(ctx);
  TRY(run_pass(ctx, "expand/" + mask_key(skip) + "/" + std::to_string(int8),
               [&] { pass_expand(ctx, skip, int8 != 0); }));
  timer_end(ctx, ti, PK_DRAFT);
  return SSD_OK;
}

// Layers a level's draft runs.
int level_depth(const ssd_model_config& c, const ssd_policy* p, int l) {
  int d = 0;
  for (uint8_t b : level_mask(c, p, l)) d += b ? 0 : 1;
  return d;
}

// The planner's level costs (fractions of a verify pass) and the number of
// levels in use at the current committed length.  cost_model 0: byte ratio;
// 1: the calibrated latency model, c_l = latency(t, depth_l, int8_l) /
// latency(t, L, 16-bit).
ssd_status planner_inputs(ssd_ctx* ctx, const ssd_policy* p, std::vector<double>& costs, int& n_active) {
  const ssd_model_config& c = ctx->cfg;
  if (p->cost_model == 0) {
    costs = level_costs(c, p);
  } else {
    for (int l = 0; l < p->n_levels; ++l)
      if (!ctx->have_beta[p->level_int8[l] ? 1 : 0] || !ctx->have_beta[0])
        return fail(ctx, SSD_ERR_STATE, "cost_model 1 needs a latency model: calibrate or set one first");
    const double full = predict_latency(ctx->beta[0], ctx->t, c.n_layers);
    if (!(full > 0.0)) return fail(ctx, SSD_ERR_STATE, "latency model predicts a non-positive verify time");
    costs.clear();
    for (int l = 0; l < p->n_levels; ++l) {
      const double v = predict_latency(ctx->beta[p->level_int8[l] ? 1 : 0], ctx->t, level_depth(c, p, l)) / full;
      if (!(v > 0.0)) return fail(ctx, SSD_ERR_STATE, "latency model predicts a non-positive draft time");
      costs.push_back(v);
    }
  }
  n_active = p->cascade_rules ? cascade_depth(c.n_layers, p->n_levels, ctx->t) : p->n_levels;
  return SSD_OK;
}

ssd_status run_plan(ssd_ctx* ctx, const ssd_policy* p, const TreePlan& plan);
ssd_status upload_plan(ssd_ctx* ctx, const TreePlan& plan);
ssd_status run_expansions(ssd_ctx* ctx, const ssd_policy* p, const TreePlan& plan);

// DyTC: plan a tree, upload it and run its expansions (drafts) in order.
ssd_status dytc_draft(ssd_ctx* ctx, const ssd_policy* p, TreePlan& plan) {
  std::vector<double> costs;
  int n_active = 0;
  TRY(planner_inputs(ctx, p, costs, n_active));
  const std::vector<double> a(ctx->ema.begin(), ctx->ema.begin() + n_active);
  costs.resize(n_active);
  plan = dytc_plan(a, costs, p->tree_max_nodes, p->tree_max_depth);
  return run_plan(ctx, p, plan);
}

// Upload a tree plan and run its draft expansions in order (each fills its children's tokens).
ssd_status run_plan(ssd_ctx* ctx, const ssd_policy* p, const TreePlan& plan) {
  TRY(upload_plan(ctx, plan));
  return run_expansions(ctx, p, plan);
}

ssd_status upload_plan(ssd_ctx* ctx, const TreePlan& plan) {
  const int n = (int)plan.parents.size();
  TRY(upload_tree(ctx, nullptr, plan.parents.data(), n));
  const int ne = (int)plan.exp_node.size();
  std::vector<int> buf(3 * kMaxRows + 1, 0);
  for (int e = 0; e < ne; ++e) {
    buf[e] = plan.exp_node[e];
    buf[kMaxRows + e] = plan.child0[e];
    buf[2 * kMaxRows + e] = plan.child1[e];
  }
  TRY(upload(ctx, ctx->P(ctx->off.exp_node), buf.data(), kMaxRows * 4));
  TRY(upload(ctx, ctx->P(ctx->off.exp_c0), buf.data() + kMaxRows, kMaxRows * 4));
  TRY(upload(ctx, ctx->P(ctx->off.exp_c1), buf.data() + 2 * kMaxRows, kMaxRows * 4));
  return SSD_OK;
}

// The plan's expansions, stream-ordered (no host synchronisation): the expansion counter is reset first.
ssd_status run_expansions(ssd_ctx* ctx, const ssd_policy* p, const TreePlan& plan) {
  CU(cudaMemsetAsync(&ctx->st()->exp_idx, 0, sizeof(int), ctx->stream));
  for (size_t e = 0; e < plan.exp_node.size(); ++e) {
    const int l = plan.exp_level[e];
    TRY(launch_expand(ctx, level_mask(ctx->cfg, p, l), p->level_int8[l]));
  }
  return SSD_OK;
}

ssd_status validate_policy(ssd_ctx* ctx, const ssd_policy* p) {
  if (!p) return fail(ctx, SSD_ERR_INVALID_ARG, "policy is null");
  const int L = ctx->cfg.n_layers;
  switch (p->kind) {
    case SSD_POLICY_AR:
      return SSD_OK;
    case SSD_POLICY_STATIC:
      if (!p->skip_mask) return fail(ctx, SSD_ERR_INVALID_ARG, "STATIC policy needs skip_mask");
      // fallthrough
    case SSD_POLICY_CLASP:
      if (p->draft_k < 1 || p->draft_k + 1 > ctx->cfg.max_rows)
        return fail(ctx, SSD_ERR_INVALID_ARG, "draft_k must be in [1, max_rows-1]");
      if (!isfinite(p->draft_exit)) return fail(ctx, SSD_ERR_INVALID_ARG, "draft_exit must be finite");
      if (p->early_exit < 0 || p->early_exit > L) return fail(ctx, SSD_ERR_INVALID_ARG, "early_exit must be in [0, L]");
      if (p->kind == SSD_POLICY_CLASP) {
        if (p->dp_n_skip < 0 || p->dp_n_skip > L || p->dp_n_skip + 1 > ctx->cfg.max_rows)
          return fail(ctx, SSD_ERR_INVALID_ARG, "dp_n_skip out of range");
        if (p->dp_interval < 0) return fail(ctx, SSD_ERR_INVALID_ARG, "dp_interval < 0");
      }
      return SSD_OK;
    case SSD_POLICY_DYTC:
    case SSD_POLICY_HCASCADE:
    case SSD_POLICY_VCASCADE: {
      if (p->n_levels < 1 || p->n_levels > 3 || !p->level_skip || !p->level_int8)
        return fail(ctx, SSD_ERR_INVALID_ARG, "DYTC and HCASCADE need 1..3 levels");
      if (p->kind == SSD_POLICY_VCASCADE) {
        if (p->vc_lo < 0 || p->vc_lo >= p->vc_hi || p->vc_hi >= p->n_levels)
          return fail(ctx, SSD_ERR_INVALID_ARG, "need 0 <= vc_lo < vc_hi < n_levels");
        if (p->draft_k < 1 || p->draft_k + 1 > ctx->cfg.max_rows)
          return fail(ctx, SSD_ERR_INVALID_ARG, "draft_k must be in [1, max_rows-1]");
      } else if (p->kind == SSD_POLICY_HCASCADE) {
        if (!p->hc_len) return fail(ctx, SSD_ERR_INVALID_ARG, "HCASCADE needs hc_len");
        int k = 0;
        for (int l = 0; l < p->n_levels; ++l) {
          if (p->hc_len[l] < 0) return fail(ctx, SSD_ERR_INVALID_ARG, "hc_len must be >= 0");
          k += p->hc_len[l];
        }
        if (k < 1 || k > 63 || k + 1 > ctx->cfg.max_rows)
          return fail(ctx, SSD_ERR_INVALID_ARG, "sum(hc_len) must be in [1, min(63, max_rows - 1)]");
      } else {
        if (p->tree_max_nodes < 1 || p->tree_max_nodes + 1 > ctx->cfg.max_rows || p->tree_max_nodes > 63)
          return fail(ctx, SSD_ERR_INVALID_ARG, "tree_max_nodes out of range");
        if (p->tree_max_depth < 1) return fail(ctx, SSD_ERR_INVALID_ARG, "tree_max_depth < 1");
      }
      if (p->cost_model != 0 && p->cost_model != 1) return fail(ctx, SSD_ERR_INVALID_ARG, "cost_model must be 0 or 1");
      if (p->level_exit)
        for (int l = 0; l < p->n_levels; ++l)
          if (p->level_exit[l] < 0 || p->level_exit[l] > L)
            return fail(ctx, SSD_ERR_INVALID_ARG, "level_exit must be in [0, L]");
      for (int l = 0; l + 1 < p->n_levels; ++l) {
        const std::vector<uint8_t> lo = level_mask(ctx->cfg, p, l), hi = level_mask(ctx->cfg, p, l + 1);
        for (int i = 0; i < L; ++i)
          if (hi[i] && !lo[i])
            return fail(ctx, SSD_ERR_INVALID_ARG, "DYTC levels must be nested (higher level keeps a superset)");
      }
      return SSD_OK;
    }
    default:
      return fail(ctx, SSD_ERR_INVALID_ARG, "unknown policy kind");
  }
}

}  // namespace

// ============================================================================ C ABI

extern "C" {

size_t ssd_workspace_bytes(const ssd_model_config* cfg) {
  if (!config_ok(cfg)) return 0;
  return layout_of(*cfg).total;
}

int ssd_weight_count(const ssd_model_config* cfg) { return config_ok(cfg) ? 3 + 6 * cfg->n_layers : -1; }

ssd_status ssd_create(const ssd_model_config* cfg, void* workspace, size_t ws_bytes, void* cuda_stream,
                      ssd_ctx** out) {
  if (!out) return SSD_ERR_INVALID_ARG;
  *out = nullptr;
  if (!config_ok(cfg) || !workspace) return SSD_ERR_INVALID_ARG;
  if (((uintptr_t)workspace) & 255) return SSD_ERR_INVALID_ARG;
  Offsets off = layout_of(*cfg);
  if (ws_bytes < off.total) return SSD_ERR_CAPACITY;
  ssd_ctx* ctx = new (std::nothrow) ssd_ctx();
  if (!ctx) return SSD_ERR_OOM;
  ctx->cfg = *cfg;
  ctx->off = off;
  ctx->ws = (char*)workspace;
  ctx->stream = (cudaStream_t)cuda_stream;
  if (cudaStreamCreateWithFlags(&ctx->side, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    delete ctx;
    return SSD_ERR_CUDA;
  }
  ctx->fp16 = cfg->dtype == SSD_FP16;
  ctx->cur_skip.assign(cfg->n_layers, 0);
  cudaGetDevice(&ctx->device);
  cudaDeviceGetAttribute(&ctx->sms, cudaDevAttrMultiProcessorCount, ctx->device);
  // stream-K partial tiles of the tcgen05 projection: two per CTA (one CTA per SM), 2 x 64 x 128 floats each
  if ((size_t)ctx->sms * 2 * 2 * 64 * 128 * 4 > kMmaPart) {
    cudaStreamDestroy(ctx->side);
    delete ctx;
    return SSD_ERR_INVALID_ARG;
  }
  if (!init_kernels()) {
    cudaGetLastError();
    delete ctx;
    return SSD_ERR_CUDA;
  }
  ctx->h_pin_n = 1 << 20;
  if (cudaMallocHost(&ctx->h_pin, ctx->h_pin_n) != cudaSuccess) {
    delete ctx;
    return SSD_ERR_OOM;
  }
  // zero the small state + counters, identity block table, RoPE table
  ssd_status s = SSD_OK;
  do {
    if (cudaMemsetAsync(ctx->P(off.st), 0, off.rope_cos - off.st, ctx->stream) != cudaSuccess) {
      s = SSD_ERR_CUDA;
      break;
    }
    if (cudaMemsetAsync(ctx->P(off.mma_cnt), 0, 4096 * 4, ctx->stream) != cudaSuccess) {
      s = SSD_ERR_CUDA;
      break;
    }
    const std::vector<float> ones(64, 1.0f);
    if (cudaMemcpy(ctx->P(off.mma_ones), ones.data(), 64 * 4, cudaMemcpyHostToDevice) != cudaSuccess) {
      s = SSD_ERR_CUDA;
      break;
    }
    const int half = cfg->head_dim / 2, pages = n_pages_of(*cfg);
    std::vector<float> cs((size_t)cfg->max_ctx * half), sn((size_t)cfg->max_ctx * half);
    for (int p = 0; p < cfg->max_ctx; ++p)
      for (int i = 0; i < half; ++i) {
        const double inv = pow((double)cfg->rope_base, -(2.0 * i) / (double)cfg->head_dim);
        const double ang = (double)p * inv;
        cs[(size_t)p * half + i] = (float)cos(ang);
        sn[(size_t)p * half + i] = (float)sin(ang);
      }
    std::vector<int> bt(pages);
    for (int i = 0; i < pages; ++i) bt[i] = i;
    if (cudaMemcpy(ctx->P(off.rope_cos), cs.data(), cs.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(ctx->P(off.rope_sin), sn.data(), sn.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(ctx->P(off.btab), bt.data(), bt.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess) {
      s = SSD_ERR_CUDA;
      break;
    }
    DevState st0{};
    st0.gen_cap = 0;
    if (cudaMemcpy(ctx->P(off.st), &st0, sizeof(st0), cudaMemcpyHostToDevice) != cudaSuccess) s = SSD_ERR_CUDA;
    if (cudaStreamSynchronize(ctx->stream) != cudaSuccess) s = SSD_ERR_CUDA;
  } while (0);
  if (s != SSD_OK) {
    cudaFreeHost(ctx->h_pin);
    delete ctx;
    return s;
  }
  *out = ctx;
  return SSD_OK;
}

ssd_status ssd_load_weights(ssd_ctx* ctx, const void* const* p, int n) {
  if (!ctx) return SSD_ERR_INVALID_ARG;
  const int L = ctx->cfg.n_layers;
  if (!p || n != 3 + 6 * L) return fail(ctx, SSD_ERR_INVALID_ARG, "expected 3 + 6 * n_layers weight pointers");
  for (int i = 0; i < n; ++i)
    if (!p[i] || ((uintptr_t)p[i] & 15)) return fail(ctx, SSD_ERR_INVALID_ARG, "weight pointer null or not 16-byte aligned");
  ctx->embed = p[0];
  ctx->final_norm = p[1];
  ctx->lm_head = p[2];
  ctx->layers.resize(L);
  for (int i = 0; i < L; ++i) {
    const void* const* q = p + 3 + 6 * i;
    ctx->layers[i] = LayerW{q[0], q[1], q[2], q[3], q[4], q[5]};
  }
  drop_graphs(ctx);
  ctx->weights = true;
  return SSD_OK;
}

ssd_status ssd_set_option(ssd_ctx* ctx, int option, int value) {
  if (!ctx) return SSD_ERR_INVALID_ARG;
  switch (option) {
    case SSD_OPT_GEMM_IMPL:
#ifdef SSD_CROSSCHECK
      if (value < 0 || value > 5) return fail(ctx, SSD_ERR_INVALID_ARG, "GEMM_IMPL is 0..5");
#else
      if (value != 0)
        return fail(ctx, SSD_ERR_INVALID_ARG, "GEMM_IMPL 1..3 selects cross-check kernels of the test library only");
#endif
      ctx->gemm_impl = value;
      break;
    case SSD_OPT_USE_GRAPHS:
      ctx->use_graphs = value != 0;
      break;
    case SSD_OPT_TIMING:
      ctx->timing = value != 0;
      break;
    case SSD_OPT_PDL:
      ctx->use_pdl = value != 0;
      break;
    case SSD_OPT_TRACE:
      ctx->tracing = value != 0;
      break;
    case SSD_OPT_CYCLE_LOG:
      ctx->cycle_log = value != 0;
      ctx->log.clear();
      return SSD_OK;  // host-side only: the captured passes stay valid
    case SSD_OPT_L2_PREFETCH_MB:
      if (value < 0 || value > 96) return fail(ctx, SSD_ERR_INVALID_ARG, "L2 prefetch is 0..96 MB");
      ctx->pf_cap = (size_t)value << 20;
      break;
    default:
      return fail(ctx, SSD_ERR_INVALID_ARG, "unknown option");
  }
  drop_graphs(ctx);
  return SSD_OK;
}

ssd_status ssd_prefill(ssd_ctx* ctx, const int32_t* tokens, int n, int32_t* next_token) {
  if (!ctx) return SSD_ERR_INVALID_ARG;
  if (!ctx->weights) return fail(ctx, SSD_ERR_STATE, "no weights loaded");
  if (!tokens || n < 1) return fail(ctx, SSD_ERR_INVALID_ARG, "need at least one token");
  for (int i = 0; i < n; ++i)
    if (tokens[i] < 0 || tokens[i] >= ctx->cfg.vocab) return fail(ctx, SSD_ERR_INVALID_ARG, "token id out of range");
  int t0 = ctx->t;
  if (ctx->have_pending) {
    // the pending token is not in the cache; prefill continues after the committed prefix
  }
  if (t0 + n + 1 > ctx->cfg.max_ctx) return fail(ctx, SSD_ERR_CAPACITY, "prompt exceeds max_ctx");
  TRY(upload(ctx, ctx->P(ctx->off.prompt), tokens, (size_t)n * 4));
  const int chunk = ctx->cfg.max_rows;
  g_pdl = ctx->use_pdl != 0;
  const long long before = g_launches;
  for (int off = 0; off < n; off += chunk) {
    const int m = std::min(chunk, n - off);
    pass_prefill_chunk(ctx, off, m, off + m == n);
  }
  ctx->launches += g_launches - before;
  CU(cudaGetLastError());
  DevState s;
  TRY(read_state(ctx, &s));
  ctx->have_pending = true;
  ctx->have_target = true;
  if (next_token) *next_token = s.pending;
  return SSD_OK;
}

ssd_status ssd_decode_ar(ssd_ctx* ctx, int n, int32_t* out_tokens) {
  if (!ctx) return SSD_ERR_INVALID_ARG;
  if (!need_state(ctx)) return fail(ctx, SSD_ERR_STATE, "prefill first");
  if (n < 0) return fail(ctx, SSD_ERR_INVALID_ARG, "n < 0");
  if (ctx->t + n + 1 > ctx->cfg.max_ctx) return fail(ctx, SSD_ERR_CAPACITY, "would exceed max_ctx");
  int z[2] = {0, n};
  TRY(upload(ctx, &ctx->st()->gen_count, z, 8));
  int* out = ctx->P<int>(ctx->off.out_tokens);
  for (int i = 0; i < n; ++i) TRY(launch_ar(ctx, out));
  ctx->ar_steps += n;
  if (out_tokens && n) TRY(d2h(ctx, out_tokens, out, (size_t)n * 4));
  DevState s;
  TRY(read_state(ctx, &s));
  return SSD_OK;
}

ssd_status ssd_draft(ssd_ctx* ctx, const uint8_t* skip_mask, int act_int8, int k, float exit_threshold,
                     int32_t* out_draft, int32_t* n_drafted) {
  if (!ctx) return SSD_ERR_INVALID_ARG;
  if (!need_state(ctx)) return fail(ctx, SSD_ERR_STATE, "prefill first");
  TRY(check_skip(ctx, skip_mask));
  if (k < 1 || k + 1 > ctx->cfg.max_rows) return fail(ctx, SSD_ERR_INVALID_ARG, "k must be in [1, max_rows-1]");
  if (!isfinite(exit_threshold)) return fail(ctx, SSD_ERR_INVALID_ARG, "exit_threshold must be finite");
  if (ctx->t + k + 1 > ctx->cfg.max_ctx) return fail(ctx, SSD_ERR_CAPACITY, "would exceed max_ctx");
  std::vector<uint8_t> m(skip_mask, skip_mask + ctx->cfg.n_layers);
  for (auto& b : m) b = b ? 1 : 0;
  TRY(launch_draft(ctx, m, act_int8 ? 1 : 0, k, exit_threshold));
  if (out_draft) TRY(d2h(ctx, out_draft, ctx->P(ctx->off.drafts), (size_t)k * 4));
  int n = k;
  if (exit_threshold > 0.f) {
    DevState s;
    TRY(read_state(ctx, &s));
    n = s.draft_n;
  }
  TRY(sync(ctx));
  if (n_drafted) *n_drafted = n;
  return SSD_OK;
}

ssd_status ssd_verify(ssd_ctx* ctx, const int32_t* tokens, const int32_t* parents, int n, int32_t* accepted_len,
                      int32_t* accepted_path, int32_t* bonus) {
  if (!ctx) return SSD_ERR_INVALID_ARG;
  if (!need_state(ctx)) return fail(ctx, SSD_ERR_STATE, "prefill first");
  if (!tokens || n < 1 || n > ctx->cfg.max_rows) return fail(ctx, SSD_ERR_INVALID_ARG, "n must be in [1, max_rows]");
  if (parents && n > 63) return fail(ctx, SSD_ERR_INVALID_ARG, "trees hold at most 63 nodes");
  for (int i = 0; i < n; ++i)
    if (tokens[i] < 0 || tokens[i] >= ctx->cfg.vocab) return fail(ctx, SSD_ERR_INVALID_ARG, "token id out of range");
  if (tokens[0] != ctx->pending) return fail(ctx, SSD_ERR_INVALID_ARG, "tokens[0] must be the pending token");
  if (parents) TRY(validate_tree(ctx, parents, n));
  if (ctx->t + n + 1 > ctx->cfg.max_ctx) return fail(ctx, SSD_ERR_CAPACITY, "would exceed max_ctx");
  if (parents) {
    TRY(upload_tree(ctx, tokens, parents, n));
  } else if (n > 1) {
    TRY(upload(ctx, ctx->P(ctx->off.drafts), tokens + 1, (size_t)(n - 1) * 4));
  }
  TRY(launch_verify(ctx, n, parents != nullptr, nullptr));
  DevState s;
  TRY(read_state(ctx, &s));
  if (accepted_len) *accepted_len = s.n_acc;
  if (bonus) *bonus = s.bonus;
  if (accepted_path)
    for (int i = 0; i <= s.n_acc; ++i) accepted_path[i] = s.path[i];
  ctx->have_target = true;
  return SSD_OK;
}

ssd_status ssd_rollback(ssd_ctx* ctx, int new_len, int32_t pending_token) {
  if (!ctx) return SSD_ERR_INVALID_ARG;
  if (new_len < 0 || new_len > ctx->t) return fail(ctx, SSD_ERR_INVALID_ARG, "new_len must be in [0, t]");
  if (pending_token >= ctx->cfg.vocab) return fail(ctx, SSD_ERR_INVALID_ARG, "pending token out of range");
  int v[2] = {new_len, pending_token >= 0 ? pending_token : ctx->pending};
  TRY(upload(ctx, ctx->st(), v, 8));
  TRY(sync(ctx));
  ctx->t = new_len;
  if (pending_token >= 0) {
    ctx->pending = pending_token;
    ctx->have_pending = true;
  }
  // the CLaSp target survives while its token stays committed (its states are in the stash)
  ctx->have_target = ctx->have_target && ctx->tgt_pos >= 0 && ctx->tgt_pos < new_len;
  return SSD_OK;
}

ssd_status ssd_dp_select(ssd_ctx* ctx, int n_skip, uint8_t* mask_out, float* value_out) {
  if (!ctx) return SSD_ERR_INVALID_ARG;
  if (!ctx->weights) return fail(ctx, SSD_ERR_STATE, "no weights loaded");
  if (!ctx->have_target) return fail(ctx, SSD_ERR_STATE, "no CLaSp target: prefill or verify first");
  const int L = ctx->cfg.n_layers;
  if (n_skip < 0 || n_skip > L || n_skip + 1 > ctx->cfg.max_rows)
    return fail(ctx, SSD_ERR_INVALID_ARG, "n_skip must be in [0, L] and n_skip + 1 <= max_rows");
  if (ctx->t + n_skip + 1 > ctx->cfg.max_ctx) return fail(ctx, SSD_ERR_CAPACITY, "no scratch slots left");
  TRY(launch_dp(ctx, n_skip));
  std::vector<uint8_t> m(L);
  float v = 0.f;
  TRY(d2h(ctx, m.data(), ctx->P(ctx->off.dp_mask), L));
  TRY(d2h(ctx, &v, ctx->P(ctx->off.dp_value), 4));
  TRY(sync(ctx));
  ctx->cur_skip = m;
  ctx->last_dp_n = n_skip;
  if (mask_out) memcpy(mask_out, m.data(), L);
  if (value_out) *value_out = v;
  if (ctx->cycle_log) {
    ssd_cycle_record r;
    memset(&r, 0, sizeof(r));
    r.kind = 2;
    r.t = ctx->t;
    memcpy(r.mask, m.data(), L);
    r.dp_value = v;
    ctx->log.push_back(r);
  }
  return SSD_OK;
}

ssd_status ssd_get_dp_table(ssd_ctx* ctx, int* n_skip_out, float* val_out, uint8_t* back_out) {
  if (!ctx) return SSD_ERR_INVALID_ARG;
  if (ctx->last_dp_n < 0) return fail(ctx, SSD_ERR_STATE, "no DP search has run");
  const int L = ctx->cfg.n_layers, n = ctx->last_dp_n, ncol = ctx->cfg.max_rows;
  std::vector<float> v((size_t)(L + 1) * ncol);
  std::vector<uint8_t> b((size_t)(L + 1) * ncol);
  TRY(d2h(ctx, v.data(), ctx->P(ctx->off.dp_val), v.size() * 4));
  TRY(d2h(ctx, b.data(), ctx->P(ctx->off.dp_back), b.size()));
  TRY(sync(ctx));
  for (int i = 0; i <= L; ++i)
    for (int j = 0; j <= n; ++j) {
      int lo, hi;
      dp_range(L, n, i, lo, hi);
      const bool in = j >= lo && j <= hi;
      if (val_out) val_out[(size_t)i * (n + 1) + j] = in ? v[(size_t)i * ncol + j] : NAN;
      if (back_out) back_out[(size_t)i * (n + 1) + j] = in ? b[(size_t)i * ncol + j] : 255;
    }
  if (n_skip_out) *n_skip_out = n;
  return SSD_OK;
}

ssd_status ssd_get_cycle_log(ssd_ctx* ctx, ssd_cycle_record* out, int max_records, int* n_records) {
  if (!ctx || !n_records || max_records < 0 || (max_records > 0 && !out)) return SSD_ERR_INVALID_ARG;
  const int n = std::min<int>(max_records, (int)ctx->log.size());
  if (n) memcpy(out, ctx->log.data(), (size_t)n * sizeof(ssd_cycle_record));
  *n_records = n;
  return SSD_OK;
}

ssd_status ssd_set_ema(ssd_ctx* ctx, const double* ema, int n_levels) {
  if (!ctx) return SSD_ERR_INVALID_ARG;
  if (!ema || n_levels < 1 || n_levels > 3) return fail(ctx, SSD_ERR_INVALID_ARG, "need 1..3 estimates");
  for (int l = 0; l < n_levels; ++l)
    if (!(ema[l] >= 0.0 && ema[l] <= 1.0)) return fail(ctx, SSD_ERR_INVALID_ARG, "estimates must be in [0, 1]");
  ctx->ema.assign(ema, ema + n_levels);
  return SSD_OK;
}

int ssd_cascade_depth(int n_layers, int n_levels, int seq_len) { return cascade_depth(n_layers, n_levels, seq_len); }

void ssd_abi_sizes(size_t* out, int n) {
  const size_t sz[5] = {sizeof(ssd_model_config), sizeof(ssd_policy), sizeof(ssd_stats), sizeof(ssd_attention_args),
                        sizeof(ssd_cycle_record)};
  for (int i = 0; i < n && i < 5; ++i) out[i] = sz[i];
}

namespace {
ssd_status copy_plan(const TreePlan& plan, int32_t* parents_out, int* n_nodes, int32_t* exp_node_out,
                     int32_t* exp_level_out, int* n_exp) {
  if (plan.parents.size() > 64 || plan.exp_node.size() > 64) return SSD_ERR_CAPACITY;
  for (size_t c = 0; c < plan.parents.size(); ++c) parents_out[c] = plan.parents[c];
  for (size_t e = 0; e < plan.exp_node.size(); ++e) {
    exp_node_out[e] = plan.exp_node[e];
    exp_level_out[e] = plan.exp_level[e];
  }
  *n_nodes = (int)plan.parents.size();
  *n_exp = (int)plan.exp_node.size();
  return SSD_OK;
}
}  // namespace

ssd_status ssd_plan_tree(int n_levels, const double* ema, const double* cost, int max_nodes, int max_depth,
                         int32_t* parents_out, int* n_nodes, int32_t* exp_node_out, int32_t* exp_level_out,
                         int* n_exp) {
  if (n_levels < 1 || n_levels > 3 || !ema || !cost || !parents_out || !n_nodes || !exp_node_out ||
      !exp_level_out || !n_exp || max_nodes < 1 || max_nodes > 63 || max_depth < 1)
    return SSD_ERR_INVALID_ARG;
  for (int l = 0; l < n_levels; ++l)
    if (!(cost[l] > 0.0) || !(ema[l] >= 0.0 && ema[l] <= 1.0)) return SSD_ERR_INVALID_ARG;
  const std::vector<double> a(ema, ema + n_levels), c(cost, cost + n_levels);
  return copy_plan(dytc_plan(a, c, max_nodes, max_depth), parents_out, n_nodes, exp_node_out, exp_level_out, n_exp);
}

ssd_status ssd_plan_hcascade(int n_levels, const int32_t* hc_len, int32_t* parents_out, int* n_nodes,
                             int32_t* exp_node_out, int32_t* exp_level_out, int* n_exp) {
  if (n_levels < 1 || n_levels > 3 || !hc_len || !parents_out || !n_nodes || !exp_node_out || !exp_level_out ||
      !n_exp)
    return SSD_ERR_INVALID_ARG;
  int k = 0;
  for (int l = 0; l < n_levels; ++l) {
    if (hc_len[l] < 0) return SSD_ERR_INVALID_ARG;
    k += hc_len[l];
  }
  if (k < 1 || k > 63) return SSD_ERR_INVALID_ARG;
  return copy_plan(hcascade_plan(hc_len, n_levels), parents_out, n_nodes, exp_node_out, exp_level_out, n_exp);
}

ssd_status ssd_fit_latency(int n, const double* seq_len, const double* depth, const double* ms, double* beta_out) {
  if (n < 3 || !seq_len || !depth || !ms || !beta_out) return SSD_ERR_INVALID_ARG;
  return fit_latency(n, seq_len, depth, ms, beta_out) ? SSD_OK : SSD_ERR_INVALID_ARG;
}

ssd_status ssd_set_latency_model(ssd_ctx* ctx, int act_int8, const double* beta) {
  if (!ctx) return SSD_ERR_INVALID_ARG;
  if (!beta) return fail(ctx, SSD_ERR_INVALID_ARG, "beta is null");
  for (int i = 0; i < 3; ++i)
    if (!isfinite(beta[i])) return fail(ctx, SSD_ERR_INVALID_ARG, "beta must be finite");
  const int m = act_int8 ? 1 : 0;
  for (int i = 0; i < 3; ++i) ctx->beta[m][i] = beta[i];
  ctx->have_beta[m] = true;
  return SSD_OK;
}

namespace {
struct EventPair {
  cudaEvent_t a = nullptr, b = nullptr;
  ~EventPair() {
    if (a) cudaEventDestroy(a);
    if (b) cudaEventDestroy(b);
  }
};
}  // namespace

ssd_status ssd_calibrate_latency(ssd_ctx* ctx, int act_int8, const int32_t* depths, int n_depths,
                                 const int32_t* seq_lens, int n_seq, int reps, const uint8_t* train, double* beta_out,
                                 double* times_ms) {
  if (!ctx) return SSD_ERR_INVALID_ARG;
  if (!need_state(ctx)) return fail(ctx, SSD_ERR_STATE, "prefill first");
  const int L = ctx->cfg.n_layers;
  if (!depths || !seq_lens || !beta_out || n_depths < 1 || n_seq < 1 || reps < 1 || reps > 1000)
    return fail(ctx, SSD_ERR_INVALID_ARG, "need depths, seq_lens, beta_out and 1 <= reps <= 1000");
  for (int j = 0; j < n_depths; ++j)
    if (depths[j] < 0 || depths[j] > L) return fail(ctx, SSD_ERR_INVALID_ARG, "depths must be in [0, L]");
  for (int i = 0; i < n_seq; ++i)
    if (seq_lens[i] < 1 || seq_lens[i] > ctx->t || seq_lens[i] + 2 > ctx->cfg.max_ctx)
      return fail(ctx, SSD_ERR_INVALID_ARG, "seq_lens must be in [1, committed length]");
  EventPair ev;
  CU(cudaEventCreate(&ev.a));
  CU(cudaEventCreate(&ev.b));
  std::vector<int> order(n_seq);
  for (int i = 0; i < n_seq; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return seq_lens[x] > seq_lens[y]; });
  std::vector<double> t_ms((size_t)n_seq * n_depths);
  std::vector<float> v(reps);
  for (int i : order) {
    TRY(ssd_rollback(ctx, seq_lens[i], -1));  // longest context first: later points only shorten it
    for (int j = 0; j < n_depths; ++j) {
      const int d = depths[j];
      std::vector<uint8_t> mask(L, 1);
      for (int m = 0; m < d; ++m) mask[(int)(((2LL * m + 1) * L) / (2LL * d))] = 0;  // d evenly spaced layers run
      TRY(launch_draft(ctx, mask, act_int8 ? 1 : 0, 1));  // builds the pass's graph once
      TRY(sync(ctx));
      for (int r = 0; r < reps; ++r) {
        CU(cudaEventRecord(ev.a, ctx->stream));
        TRY(launch_draft(ctx, mask, act_int8 ? 1 : 0, 1));
        CU(cudaEventRecord(ev.b, ctx->stream));
        CU(cudaEventSynchronize(ev.b));
        CU(cudaEventElapsedTime(&v[r], ev.a, ev.b));
      }
      std::sort(v.begin(), v.end());
      t_ms[(size_t)i * n_depths + j] = reps % 2 ? v[reps / 2] : 0.5 * ((double)v[reps / 2 - 1] + v[reps / 2]);
    }
  }
  DevState st;
  TRY(read_state(ctx, &st));
  std::vector<double> xs, xd, y;
  for (int i = 0; i < n_seq; ++i)
    for (int j = 0; j < n_depths; ++j)
      if (!train || train[(size_t)i * n_depths + j]) {
        xs.push_back(seq_lens[i]);
        xd.push_back(depths[j]);
        y.push_back(t_ms[(size_t)i * n_depths + j]);
      }
  double beta[3];
  if (!fit_latency((int)y.size(), xs.data(), xd.data(), y.data(), beta))
    return fail(ctx, SSD_ERR_INVALID_ARG, "the training points must span two sequence lengths and two depths");
  if (times_ms) memcpy(times_ms, t_ms.data(), t_ms.size() * sizeof(double));
  memcpy(beta_out, beta, sizeof(beta));
  memcpy(ctx->beta[act_int8 ? 1 : 0], beta, sizeof(beta));
  ctx->have_beta[act_int8 ? 1 : 0] = true;
  return SSD_OK;
}

ssd_status ssd_get_level_costs(ssd_ctx* ctx, const ssd_policy* p, double* costs_out, int* n_active_out) {
  if (!ctx) return SSD_ERR_INVALID_ARG;
  TRY(validate_policy(ctx, p));
  if (p->kind != SSD_POLICY_DYTC) return fail(ctx, SSD_ERR_INVALID_ARG, "policy must be DYTC");
  std::vector<double> costs;
  int n_active = 0;
  TRY(planner_inputs(ctx, p, costs, n_active));
  if (costs_out)
    for (int l = 0; l < p->n_levels; ++l) costs_out[l] = costs[l];
  if (n_active_out) *n_active_out = n_active;
  return SSD_OK;
}

ssd_status ssd_draft_tree(ssd_ctx* ctx, const ssd_policy* p, int32_t* tokens, int32_t* parents, int* n_nodes) {
  if (!ctx) return SSD_ERR_INVALID_ARG;
  if (!need_state(ctx)) return fail(ctx, SSD_ERR_STATE, "prefill first");
  if (!tokens || !parents || !n_nodes) return fail(ctx, SSD_ERR_INVALID_ARG, "null output");
  TRY(validate_policy(ctx, p));
  if (p->kind != SSD_POLICY_DYTC) return fail(ctx, SSD_ERR_INVALID_ARG, "policy must be DYTC");
  if (ctx->t + p->tree_max_nodes + 2 > ctx->cfg.max_ctx) return fail(ctx, SSD_ERR_CAPACITY, "would exceed max_ctx");
  if ((int)ctx->ema.size() != p->n_levels) ctx->ema.assign(p->n_levels, p->ema_init);
  TreePlan plan;
  TRY(dytc_draft(ctx, p, plan));
  const int n = (int)plan.parents.size();
  TRY(d2h(ctx, tokens, ctx->P(ctx->off.tree_tok), (size_t)n * 4));
  TRY(sync(ctx));
  tokens[0] = ctx->pending;
  for (int c = 0; c < n; ++c) parents[c] = plan.parents[c];
  *n_nodes = n;
  return SSD_OK;
}

ssd_status ssd_generate(ssd_ctx* ctx, const ssd_policy* p, int n_gen, int32_t* out_tokens) {
  if (!ctx) return SSD_ERR_INVALID_ARG;
  if (!need_state(ctx)) return fail(ctx, SSD_ERR_STATE, "prefill first");
  if (n_gen < 1) return fail(ctx, SSD_ERR_INVALID_ARG, "n_gen < 1");
  TRY(validate_policy(ctx, p));
  const int L = ctx->cfg.n_layers;
  const int K =
      (p->kind == SSD_POLICY_STATIC || p->kind == SSD_POLICY_CLASP || p->kind == SSD_POLICY_VCASCADE) ? p->draft_k : 0;
  int hc_k = 0;
  if (p->kind == SSD_POLICY_HCASCADE)
    for (int l = 0; l < p->n_levels; ++l) hc_k += p->hc_len[l];
  const int margin = std::max({K + 1, p->kind == SSD_POLICY_DYTC ? p->tree_max_nodes + 1 : 1, hc_k + 1}) + 1 +
                     (p->kind == SSD_POLICY_CLASP ? p->dp_n_skip + 1 : 0);
  if (ctx->t + n_gen + margin > ctx->cfg.max_ctx) return fail(ctx, SSD_ERR_CAPACITY, "would exceed max_ctx");
  int z[2] = {0, n_gen - 1};
  TRY(upload(ctx, &ctx->st()->gen_count, z, 8));
  int* dout = ctx->P<int>(ctx->off.out_tokens);
  const int first = ctx->pending;
  int produced = 1;  // the pending token at entry
  if (p->kind == SSD_POLICY_AR) {
    for (int i = 1; i < n_gen; ++i) TRY(launch_ar(ctx, dout));
    ctx->ar_steps += n_gen - 1;
  } else if (p->kind == SSD_POLICY_STATIC || p->kind == SSD_POLICY_CLASP) {
    std::vector<uint8_t> skip(L);
    if (p->kind == SSD_POLICY_STATIC) {
      for (int i = 0; i < L; ++i) skip[i] = p->skip_mask[i] ? 1 : 0;
    } else {
      if (p->dp_at_start) {
        if (!ctx->have_target) return fail(ctx, SSD_ERR_STATE, "no CLaSp target");
        TRY(ssd_dp_select(ctx, p->dp_n_skip, nullptr, nullptr));
      }
      skip = ctx->cur_skip;
    }
    add_early_exit(skip, p->early_exit);
    const int act8 = p->kind == SSD_POLICY_STATIC ? (p->act_int8 ? 1 : 0) : 0;
    int since = 0;
    while (produced < n_gen) {
      int c = (n_gen - produced + K) / (K + 1);
      if (c < 1) c = 1;
      if (p->kind == SSD_POLICY_CLASP && p->dp_interval > 0) c = std::min(c, p->dp_interval - since);
      if (ctx->cycle_log) c = 1;
      const int t_before = ctx->t;
      const float thr = p->draft_exit > 0.0 ? (float)p->draft_exit : 0.f;
      for (int j = 0; j < c; ++j) {
        TRY(launch_draft(ctx, skip, act8, K, thr));
        TRY(launch_verify(ctx, K + 1, false, dout));
      }
      since += c;
      DevState s;
      TRY(read_state(ctx, &s));
      if (ctx->cycle_log) TRY(log_cycle(ctx, 0, t_before, K + 1, nullptr, s));
      produced = 1 + s.gen_count;
      if (p->kind == SSD_POLICY_CLASP && p->dp_interval > 0 && since >= p->dp_interval && produced < n_gen) {
        ctx->have_target = true;
        TRY(ssd_dp_select(ctx, p->dp_n_skip, nullptr, nullptr));
        skip = ctx->cur_skip;
        add_early_exit(skip, p->early_exit);
        since = 0;
      }
    }
    ctx->have_target = true;
  } else if (p->kind == SSD_POLICY_VCASCADE) {
    const std::vector<uint8_t> lo = level_mask(ctx->cfg, p, p->vc_lo), hi = level_mask(ctx->cfg, p, p->vc_hi);
    while (produced < n_gen) {  // as many cycles as can all be needed, then one state read
      const int c = ctx->cycle_log ? 1 : std::max(1, (n_gen - produced + K) / (K + 1));
      const int t_before = ctx->t;
      for (int j = 0; j < c; ++j) {
        TRY(launch_draft(ctx, lo, p->level_int8[p->vc_lo], K));
        TRY(launch_draft_verify(ctx, hi, p->level_int8[p->vc_hi], K));
        TRY(launch_verify(ctx, K + 1, false, dout));
      }
      DevState s;
      TRY(read_state(ctx, &s));
      if (ctx->cycle_log) TRY(log_cycle(ctx, 0, t_before, K + 1, nullptr, s));
      produced = 1 + s.gen_count;
    }
    ctx->have_target = true;
  } else if (p->kind == SSD_POLICY_HCASCADE) {
    const TreePlan plan = hcascade_plan(p->hc_len, p->n_levels);
    const int n = (int)plan.parents.size();
    TRY(upload_plan(ctx, plan));  // the same chain every cycle
    while (produced < n_gen) {      // as many cycles as can all be needed, then one state read
      const int c = ctx->cycle_log ? 1 : std::max(1, (n_gen - produced + hc_k) / (hc_k + 1));
      const int t_before = ctx->t;
      for (int j = 0; j < c; ++j) {
        TRY(run_expansions(ctx, p, plan));
        TRY(launch_verify(ctx, n, true, dout));
      }
      DevState s;
      TRY(read_state(ctx, &s));
      if (ctx->cycle_log) TRY(log_cycle(ctx, 1, t_before, n, &plan.parents, s));
      produced = 1 + s.gen_count;
    }
    ctx->have_target = true;
  } else {  // DYTC
    if ((int)ctx->ema.size() != p->n_levels) ctx->ema.assign(p->n_levels, p->ema_init);
    while (produced < n_gen) {
      TreePlan plan;
      const int t_before = ctx->t;
      TRY(dytc_draft(ctx, p, plan));
      const int n = (int)plan.parents.size();
      TRY(launch_verify(ctx, n, true, dout));
      std::vector<int> toks(n), am(n);
      TRY(d2h(ctx, toks.data(), ctx->P(ctx->off.row_tok), (size_t)n * 4));
      TRY(d2h(ctx, am.data(), ctx->P(ctx->off.am1), (size_t)n * 4));
      DevState s;
      TRY(read_state(ctx, &s));
      dytc_update(ctx->ema, p->ema_alpha, plan, toks.data(), am.data(), s.path, s.n_acc);
      if (ctx->cycle_log) TRY(log_cycle(ctx, 1, t_before, n, &plan.parents, s));
      produced = 1 + s.gen_count;
    }
    ctx->have_target = true;
  }
  CU(cudaGetLastError());
  DevState s;
  TRY(read_state(ctx, &s));
  if (out_tokens) {
    out_tokens[0] = first;
    if (n_gen > 1) {
      TRY(d2h(ctx, out_tokens + 1, dout, (size_t)(n_gen - 1) * 4));
      TRY(sync(ctx));
    }
  }
  return SSD_OK;
}

ssd_status ssd_get_logits(ssd_ctx* ctx, int row, float* out) {
  if (!ctx || !out) return SSD_ERR_INVALID_ARG;
  if (row < 0 || row >= ctx->cfg.max_rows) return fail(ctx, SSD_ERR_INVALID_ARG, "row out of range");
  TRY(d2h(ctx, out, ctx->P<float>(ctx->off.logits) + (size_t)row * ctx->cfg.vocab, (size_t)ctx->cfg.vocab * 4));
  return sync(ctx);
}

ssd_status ssd_get_draft_conf(ssd_ctx* ctx, int n, float* out) {
  if (!ctx || !out) return SSD_ERR_INVALID_ARG;
  if (n < 1 || n + 1 > ctx->cfg.max_rows) return fail(ctx, SSD_ERR_INVALID_ARG, "n must be in [1, max_rows-1]");
  DevState s;
  TRY(read_state(ctx, &s));
  for (int i = 0; i < n; ++i) out[i] = s.draft_p1[i];
  return SSD_OK;
}

ssd_status ssd_get_hidden(ssd_ctx* ctx, int layer_i, int row, float* out) {
  if (!ctx || !out) return SSD_ERR_INVALID_ARG;
  if (layer_i < 0 || layer_i > ctx->cfg.n_layers) return fail(ctx, SSD_ERR_INVALID_ARG, "layer out of range");
  if (row < 0 || row >= ctx->cfg.max_rows) return fail(ctx, SSD_ERR_INVALID_ARG, "row out of range");
  TRY(d2h(ctx, out, stash_layer(ctx, layer_i) + (size_t)row * ctx->cfg.d_model, (size_t)ctx->cfg.d_model * 4));
  return sync(ctx);
}

ssd_status ssd_get_position(const ssd_ctx* ctx, int32_t* t, int32_t* pending) {
  if (!ctx) return SSD_ERR_INVALID_ARG;
  if (t) *t = ctx->t;
  if (pending) *pending = ctx->pending;
  return SSD_OK;
}

ssd_status ssd_get_stats(ssd_ctx* ctx, ssd_stats* out) {
  if (!ctx || !out) return SSD_ERR_INVALID_ARG;
  DevState s;
  TRY(read_state(ctx, &s));
  memset(out, 0, sizeof(*out));
  out->cycles = s.cycles;
  out->drafted = s.drafted;
  out->accepted = s.accepted;
  for (int i = 0; i <= kMaxRows; ++i) out->accept_hist[i] = s.hist[i];
  out->dp_runs = ctx->dp_runs;
  out->ar_steps = ctx->ar_steps;
  for (size_t l = 0; l < ctx->ema.size() && l < 3; ++l) out->ema[l] = ctx->ema[l];
  out->kernel_launches = ctx->launches;
  out->mma_fallbacks = ctx->mma_fallbacks;
  return SSD_OK;
}

ssd_status ssd_reset_stats(ssd_ctx* ctx) {
  if (!ctx) return SSD_ERR_INVALID_ARG;
  TRY(sync(ctx));
  long long z[2 + kMaxRows + 1 + 1] = {0};  // cycles, accepted, hist[], drafted
  static_assert(offsetof(DevState, drafted) - offsetof(DevState, cycles) == sizeof(z) - sizeof(long long),
                "statistics counters must be contiguous");
  TRY(upload(ctx, &ctx->st()->cycles, z, sizeof(z)));
  TRY(sync(ctx));
  ctx->dp_runs = ctx->ar_steps = ctx->launches = 0;
  ctx->log.clear();
  for (int i = 0; i < 4; ++i) {
    ctx->pass_ms[i] = 0;
    ctx->pass_n[i] = 0;
  }
  return SSD_OK;
}

ssd_status ssd_get_pass_times(ssd_ctx* ctx, double* out_ms, int64_t* counts) {
  if (!ctx || !out_ms || !counts) return SSD_ERR_INVALID_ARG;
  TRY(sync(ctx));
  for (int i = 0; i < 4; ++i) {
    out_ms[i] = ctx->pass_ms[i];
    counts[i] = ctx->pass_n[i];
  }
  return SSD_OK;
}

size_t ssd_attention_scratch_bytes(int rows, int n_q, int n_kv, int hd) {
  if (rows < 1 || rows > kMaxRows || n_q < 1 || n_kv < 1 || n_q % n_kv || (hd != 64 && hd != 128)) return 0;
  return align_up(sizeof(PassDesc), 256);  // the row descriptor; the split merge needs no device scratch
}

ssd_status ssd_attention(const ssd_attention_args* a, void* scratch, size_t scratch_bytes, void* stream) {
  if (!a || !a->q || !a->k_cache || !a->v_cache || !a->block_table || !a->out || !scratch)
    return SSD_ERR_INVALID_ARG;
  const size_t need = ssd_attention_scratch_bytes(a->rows, a->n_q_heads, a->n_kv_heads, a->head_dim);
  if (need == 0 || a->prefix < 0 || a->base < 0 || a->layer < 0 || a->n_pages < 1 || ((uintptr_t)scratch & 255))
    return SSD_ERR_INVALID_ARG;
  if (a->dtype < SSD_BF16 || a->dtype > SSD_F32) return SSD_ERR_INVALID_ARG;
  if (((uintptr_t)a->k_cache | (uintptr_t)a->v_cache | (uintptr_t)a->q | (uintptr_t)a->out) & 15)
    return SSD_ERR_INVALID_ARG;  // 16-byte vector and TMA accesses
  if ((int64_t)a->prefix > (int64_t)a->n_pages * kPage || (int64_t)a->base + a->rows > (int64_t)a->n_pages * kPage)
    return SSD_ERR_INVALID_ARG;
  if (scratch_bytes < need) return SSD_ERR_CAPACITY;
  PassDesc d{};
  d.rows = a->rows;
  d.prefix = a->prefix;
  d.base = a->base;
  for (int r = 0; r < a->rows; ++r) d.mask[r] = a->mask[r];
  PassDesc* dd = (PassDesc*)scratch;
  cudaStream_t st = (cudaStream_t)stream;
  g_pdl = false;
  if (!launch_store_desc(d, dd, st)) return SSD_ERR_CUDA;  // by value: no host buffer outlives the call
  AttnArgs b{};
  b.desc = dd;
  b.q = a->q;
  b.kcache = a->k_cache;
  b.vcache = a->v_cache;
  b.btab = a->block_table;
  b.n_pages = a->n_pages;
  b.layer = a->layer;
  b.n_q = a->n_q_heads;
  b.n_kv = a->n_kv_heads;
  b.hd = a->head_dim;
  b.out = a->out;
  b.rows = a->rows;
  attention_layout(a->prefix + a->rows, a->rows, a->n_q_heads / a->n_kv_heads, a->n_kv_heads, a->dtype, a->head_dim, 0,
                   &b.qb, &b.n_split);
  b.max_keys = a->prefix + a->rows;
  g_pdl = false;
  if (!launch_attention(b, a->dtype, st)) return SSD_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status ssd_get_trace(ssd_ctx* ctx, int64_t* out, int max_entries, int* n_entries) {
  if (!ctx || !out || !n_entries || max_entries < 0) return SSD_ERR_INVALID_ARG;
  const int n = std::min(ctx->trace_n, max_entries);
  std::vector<unsigned long long> buf((size_t)3 * std::max(n, 1));
  if (n) TRY(d2h(ctx, buf.data(), ctx->P(ctx->off.trace), (size_t)n * 3 * 8));
  TRY(sync(ctx));
  for (int i = 0; i < n; ++i) {
    out[4 * i] = ctx->trace_kind[i];
    out[4 * i + 1] = (int64_t)~buf[3 * i];
    out[4 * i + 2] = (int64_t)~buf[3 * i + 1];
    out[4 * i + 3] = (int64_t)buf[3 * i + 2];
  }
  *n_entries = n;
  return SSD_OK;
}

const char* ssd_last_error(const ssd_ctx* ctx) { return ctx ? ctx->err.c_str() : "null context"; }

const char* ssd_status_string(ssd_status s) {
  switch (s) {
    case SSD_OK: return "ok";
    case SSD_ERR_INVALID_ARG: return "invalid argument";
    case SSD_ERR_STATE: return "call out of order";
    case SSD_ERR_CAPACITY: return "capacity exceeded";
    case SSD_ERR_OOM: return "host out of memory";
    case SSD_ERR_CUDA: return "CUDA error";
    case SSD_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

void ssd_destroy(ssd_ctx* ctx) {
  if (!ctx) return;
  cudaStreamSynchronize(ctx->stream);
  drop_graphs(ctx);
  for (auto& e : ctx->ev_pool) {
    cudaEventDestroy(e.first);
    cudaEventDestroy(e.second);
  }
  if (ctx->h_pin) cudaFreeHost(ctx->h_pin);
  if (ctx->side) cudaStreamDestroy(ctx->side);
  delete ctx;
}

}  // extern "C"
