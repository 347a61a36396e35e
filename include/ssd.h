/*
 * ssd.h -- C ABI of libssd.so: the single-GPU hot path of training-free
 * self-speculative decoding (CAS-Spec, CLaSp) for a Llama-style decoder.
 *
 * Sources, cited by page title and section:
 *   [CAS-blog]  "CAS-Spec技术：大型语言模型推理加速新方案" (intelliparadigm.com)
 *   [CAS-paper] "CAS-Spec: Cascade Adaptive Self-Speculative Decoding for
 *               On-the-Fly Lossless Inference Acceleration of LLMs" (abstract,
 *               method summary)
 *   [CLaSp]     CLaSp article (news.43b.com.cn/a/479818), sections 一..五
 *
 * General conventions
 *   - One context = one request at batch 1, bound to one CUDA stream.  A
 *     context is not thread-safe; different contexts are independent.
 *   - Device memory is allocated by the caller (e.g. with PyTorch) and
 *     borrowed: the workspace for the context's lifetime, the weights from
 *     ssd_load_weights until ssd_destroy.  The library never allocates
 *     device memory (it allocates one small pinned host staging buffer).
 *   - Host arrays are owned by the caller and only accessed during the call.
 *   - Every call enqueues work on the context's stream.  Calls that return
 *     host values synchronise that stream before returning.
 *   - Errors come back as ssd_status; nothing is thrown across the ABI.
 *     Arguments are validated on the host before any launch; a call that
 *     fails validation leaves the context unchanged.  SSD_ERR_CUDA means a
 *     CUDA call failed (the message is in ssd_last_error); the context
 *     should then be destroyed.
 *   - Greedy choices take the largest logit, the lowest id among equal ones;
 *     a NaN logit counts as -inf.
 *   - Token ids are int32 in [0, vocab).  Weights are 16-bit (bf16 or fp16,
 *     one type per model); the KV cache, activations and the residual
 *     stream are fp32.
 */
#ifndef SSD_H
#define SSD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ssd_ctx ssd_ctx;

typedef enum {
  SSD_OK = 0,
  SSD_ERR_INVALID_ARG = 1, /* bad pointer, size, token id, tree, skip mask ... */
  SSD_ERR_STATE = 2,       /* call out of order (e.g. verify before prefill, no weights) */
  SSD_ERR_CAPACITY = 3,    /* would exceed max_ctx, max_rows or the workspace */
  SSD_ERR_OOM = 4,         /* host allocation failed */
  SSD_ERR_CUDA = 5,        /* a CUDA runtime/driver call failed, or a device-side
                              check failed (a token id past the vocabulary reached
                              the embedding: row 0 was read instead) */
  SSD_ERR_TIMEOUT = 6      /* a bounded device-side wait gave up */
} ssd_status;

/* Element types: weights are SSD_BF16 or SSD_FP16; the context's KV cache is
 * always fp32; the standalone attention also accepts 16-bit caches. */
typedef enum { SSD_BF16 = 0, SSD_FP16 = 1, SSD_F32 = 2 } ssd_dtype;

/* Shape of the decoder.  head_dim must be 64 or 128; n_q_heads a multiple of
 * n_kv_heads; d_model a multiple of 64, ffn of 16; n_layers <= 128.
 * max_ctx: KV-cache capacity in tokens (committed + scratch slots).
 * max_rows: most rows one pass may carry (verify K+1, tree N+1, DP n+1,
 * prefill chunk); 1..64. */
typedef struct {
  int n_layers, d_model, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
  int dtype; /* ssd_dtype */
  float rms_eps, rope_base;
  int max_ctx, max_rows;
} ssd_model_config;

/* Bytes of device workspace a context needs (KV cache, activations, DP
 * tables, scratch).  0 if the config is invalid. */
size_t ssd_workspace_bytes(const ssd_model_config* cfg);

/* Create a context.  workspace: device pointer, 256-byte aligned, at least
 * ssd_workspace_bytes(cfg) bytes, borrowed.  cuda_stream: a cudaStream_t
 * (NULL = legacy default stream; a non-default stream is needed for CUDA
 * graph capture, which the decode calls use).  Must be called with the
 * device that owns `workspace` current. */
ssd_status ssd_create(const ssd_model_config* cfg, void* workspace, size_t ws_bytes, void* cuda_stream,
                      ssd_ctx** out);

/* Number of tensors ssd_load_weights expects: 3 + 6 * n_layers. */
int ssd_weight_count(const ssd_model_config* cfg);

/* Borrow the weight tensors (device pointers, 16-byte aligned, row-major,
 * 16-bit of the config's dtype), in this order:
 *   0 embed [vocab, d]      1 final RMSNorm gain [d]      2 lm_head [vocab, d]
 *   then for layer i, base 3 + 6 i:
 *     +0 W_qkv [(Hq + 2 Hkv) hd, d]  rows: Wq, then Wk, then Wv
 *     +1 W_o   [d, Hq hd]
 *     +2 W_gu  [2 ffn, d]            rows: W_gate, then W_up
 *     +3 W_d   [d, ffn]
 *     +4 attention RMSNorm gain [d]  +5 FFN RMSNorm gain [d]
 * The model is the decoder the drafts skip layers of ([CAS-blog] §2.1,
 * [CLaSp] §二).  Invalidates captured graphs. */
ssd_status ssd_load_weights(ssd_ctx* ctx, const void* const* dev_ptrs, int n_tensors);

/* Append n tokens to the sequence: run them through the full model in
 * causal chunks of up to max_rows rows, writing their KV into the cache.
 * *next_token (may be NULL) receives the greedy next token, which becomes
 * the pending token of the next draft/verify/decode call.  The full-model
 * residual states of the last prompt token become the CLaSp target.
 * Errors: INVALID_ARG (n < 1, bad id), CAPACITY (past max_ctx). */
ssd_status ssd_prefill(ssd_ctx* ctx, const int32_t* tokens, int n, int32_t* next_token);

/* Plain greedy autoregressive decoding: n steps of the full model on the
 * pending token ([CLaSp] §一: one token per forward).  out_tokens[0..n-1]
 * (may be NULL) receive the new tokens; out_tokens[i] is the pending token
 * after step i. */
ssd_status ssd_decode_ar(ssd_ctx* ctx, int n, int32_t* out_tokens);

/* Draft up to k tokens (1 <= k <= max_rows-1) with the layer-skipped model
 * ([CAS-blog] §2.1, [CLaSp] §三 stage 1): skip_mask[i] != 0 bypasses layer
 * i entirely (attention + FFN; no KV written for it); act_int8 != 0
 * quantizes the inputs of the seven per-layer projections per token to
 * int8 ([CAS-blog] §2.1 item 3).  Draft r runs in scratch slot t + r and
 * sees the committed prefix plus the earlier drafts.  An early exit e layers
 * before the end ([CAS-blog] §2.1 item 2) is the mask with the last e layers
 * set: the same forward.
 * Draft exit ([CLaSp] §四, the draft exit threshold): with exit_threshold
 * > 0, drafting ends after the first draft whose top-1 softmax probability
 * (fp32, from the draft's fp32 logits) is below exit_threshold; that draft
 * is kept.  exit_threshold <= 0 drafts exactly k.  *n_drafted (may be
 * NULL) receives the number of drafts n (1 <= n <= k); out_draft[0..k-1]
 * (may be NULL) receive them, entries n..k-1 are -1.  The committed
 * length does not change.  Errors: INVALID_ARG (k out of range, threshold
 * not finite), STATE (no prefill), CAPACITY (t + k + 1 > max_ctx). */
ssd_status ssd_draft(ssd_ctx* ctx, const uint8_t* skip_mask, int act_int8, int k, float exit_threshold,
                     int32_t* out_draft, int32_t* n_drafted);

/* Verify n rows in one full-model pass and accept greedily ([CLaSp] §三
 * stage 2, §一).  tokens[0] must be the pending token; tree_parents NULL
 * means a chain (row r's parent is r-1), else tree_parents[0] = -1 and
 * 0 <= tree_parents[c] < c ([CAS-paper] abstract: drafts form a tree
 * verified in one pass).  Row c runs at position t + depth(c) in slot t + c
 * and sees the committed prefix and its ancestors.  Acceptance walks from
 * the root to the child whose token equals the full model's argmax;
 * *accepted_len = n_acc, accepted_path[0..n_acc] = the accepted node ids
 * (path[0] = 0), *bonus = the argmax at the last accepted node.  The
 * accepted nodes' KV is compacted into slots t..t+n_acc, the committed
 * length becomes t + n_acc + 1 (the rest is rolled back), and the bonus
 * becomes the pending token.  accepted_path may be NULL. */
ssd_status ssd_verify(ssd_ctx* ctx, const int32_t* tokens, const int32_t* tree_parents, int n,
                      int32_t* accepted_len, int32_t* accepted_path, int32_t* bonus);

/* Truncate the committed length to new_len (0 <= new_len <= t); slots past
 * it become scratch.  If pending_token >= 0 it becomes the pending token;
 * otherwise the pending token is unchanged.  The CLaSp target (see
 * ssd_dp_select) is kept when its token is still committed (its position <
 * new_len) and dropped otherwise.  Enqueues nothing. */
ssd_status ssd_rollback(ssd_ctx* ctx, int new_len, int32_t pending_token);

/* CLaSp skip-set search ([CLaSp] §三): dp[i][j] = the best cosine similarity
 * to the target's full-model residual after i layers with j of them
 * skipped; all j of one layer run as rows of one pass that sees the
 * committed prefix and each row's own K/V only (no KV written to the
 * committed cache).  A tie keeps the layer.  The target is the last
 * accepted token of the last verify (or the last prefilled token).
 * skip_mask_out[0..L-1] (may be NULL) receives 1 for skipped layers;
 * *dp_value_out (may be NULL) receives dp[L][n_skip].  The mask is also
 * kept in the context for ssd_generate.  Errors: INVALID_ARG
 * (n_skip < 0 or > L, or n_skip + 1 > max_rows), STATE (no target yet). */
ssd_status ssd_dp_select(ssd_ctx* ctx, int n_skip, uint8_t* skip_mask_out, float* dp_value_out);

/* The whole table of the last ssd_dp_select, for checking it cell by cell:
 * val_out[i * (n + 1) + j] = dp[i][j] (the chosen state's cosine to the
 * target after i layers with j skipped) and back_out[...] = 1 if that state
 * skipped layer i-1, 0 if it kept it, for i = 0..L, j = 0..n, where n is that
 * call's n_skip (*n_skip_out).  Cells outside the searched range
 * j in [max(0, n - (L - i)), min(i, n)] get NaN and 255.  val_out and
 * back_out (either may be NULL) hold (L + 1) * (n + 1) entries.
 * Errors: STATE (no DP has run). */
ssd_status ssd_get_dp_table(ssd_ctx* ctx, int* n_skip_out, float* val_out, uint8_t* back_out);

/* Drafting policy for ssd_generate. */
typedef enum {
  SSD_POLICY_STATIC = 0,
  SSD_POLICY_CLASP = 1,
  SSD_POLICY_DYTC = 2,
  SSD_POLICY_AR = 3,
  SSD_POLICY_HCASCADE = 4, /* horizontal cascade baseline over the DYTC levels (hc_len) */
  SSD_POLICY_VCASCADE = 5  /* vertical cascade baseline over two of the DYTC levels (vc_lo, vc_hi) */
} ssd_policy_kind;

typedef struct {
  int kind;                /* ssd_policy_kind */
  int draft_k;             /* linear draft length (STATIC, CLASP) */
  int act_int8;            /* STATIC: quantize draft activations */
  const uint8_t* skip_mask;/* STATIC: [n_layers] */
  int dp_n_skip;           /* CLASP: layers to skip */
  int dp_interval;         /* CLASP: re-run the DP every this many verify steps */
  int dp_at_start;         /* CLASP: run the DP once before the first cycle */
  /* DYTC ([CAS-blog] §2.2, §3.1-3.2): up to 3 cascade levels */
  int n_levels;
  const uint8_t* level_skip;   /* [n_levels][n_layers]; nested: level l+1 keeps every layer level l keeps */
  const int32_t* level_int8;   /* [n_levels] */
  double ema_alpha, ema_init;  /* 0.2, 0.65 */
  int tree_max_nodes, tree_max_depth; /* <= 16 (and <= max_rows-1), <= 15 */
  /* STATIC, CLASP: draft exit threshold ([CLaSp] §四; the pages find ~0.7
   * best).  Each cycle's drafting ends after the first draft whose top-1
   * softmax probability is below it (that draft kept); the verify pass
   * keeps draft_k + 1 rows, the rows past the exit carrying token -1 that
   * no argmax equals.  <= 0: every cycle drafts draft_k. */
  double draft_exit;
  /* Early exit ([CAS-blog] §2.1 item 2, §2.2: L1 = 70 % sparsity + a 4-layer
   * early exit): a draft that exits e layers early runs none of the last e
   * layers (no KV written for them) and reads the lm_head after layer
   * L - e - 1, exactly as if those layers were in its skip set.
   * early_exit: STATIC, CLASP drafts (added to the static or DP skip set);
   * level_exit: DYTC, [n_levels] or NULL (none).  0 <= e <= L; the nested
   * rule for DYTC levels applies to the skip sets with the exits added. */
  int early_exit;
  const int32_t* level_exit;
  /* DYTC scheduler inputs.  cost_model 0: level cost c_l = bytes of the
   * level's pass / bytes of a full pass (batch-1 decode streams weights);
   * 1: the latency model of [CAS-blog] §3.2 set by ssd_calibrate_latency or
   * ssd_set_latency_model, c_l = latency(t, depth_l, int8_l) / latency(t, L,
   * 16-bit) at the committed length t.  cascade_rules != 0: only the first
   * ssd_cascade_depth(L, n_levels, t) levels are used. */
  int cost_model;
  int cascade_rules;
  /* HCASCADE ([CAS-paper] abstract: the classic horizontal cascade DyTC is
   * compared with): each cycle drafts a chain whose first hc_len[n_levels-1]
   * positions come from the highest level, the next hc_len[n_levels-2] from
   * the level below, ..., the last hc_len[0] from L1, then verifies it in one
   * pass.  Uses n_levels, level_skip, level_int8, level_exit (nested as for
   * DYTC); 1 <= sum(hc_len) <= min(63, max_rows - 1). */
  const int32_t* hc_len;
  /* VCASCADE (the classic vertical cascade: a draft model's own drafts come
   * from a smaller draft): each cycle level vc_lo drafts draft_k tokens,
   * level vc_hi checks them in one multi-row pass and keeps the prefix it
   * agrees with plus its correction of the first one it rejects, and the
   * target verifies that chain.  0 <= vc_lo < vc_hi < n_levels (vc_hi runs a
   * superset of vc_lo's layers). */
  int vc_lo, vc_hi;
} ssd_policy;

typedef struct {
  int64_t cycles, drafted, accepted, generated, dp_runs, ar_steps;
  int64_t accept_hist[65]; /* cycles that accepted exactly i drafts */
  double ema[3];           /* DyTC acceptance estimates after the last cycle */
  int64_t kernel_launches; /* kernels this context launched (graph nodes counted per replay) */
  int64_t mma_fallbacks;   /* multi-row projections the tcgen05 kernel refused; each failed its pass with
                              SSD_ERR_CUDA (there is no other kernel for them); 0 in normal operation */
} ssd_stats;

/* One entry of the per-cycle log that ssd_generate keeps while SSD_OPT_CYCLE_LOG
 * is on (and ssd_dp_select adds a DP entry to).  Logging makes ssd_generate
 * read the device state after every cycle (it otherwise runs several cycles
 * per read); it is meant for checking a generation step by step. */
typedef struct {
  int32_t kind;         /* 0 linear cycle (STATIC, CLASP, VCASCADE), 1 tree cycle (DYTC, HCASCADE),
                           2 CLaSp DP run */
  int32_t t;            /* committed length before the cycle */
  int32_t n_rows;       /* verify rows: pending token + drafts (linear), tree nodes (tree) */
  int32_t n_acc, bonus; /* accepted drafts, bonus token */
  int32_t tokens[64];   /* token of each verify row (-1 for rows past a draft exit) */
  int32_t parents[64];  /* tree: parent of each node, parents[0] = -1; linear: r - 1 */
  int32_t argmax[64];   /* the full model's greedy token at each verify row */
  int32_t path[65];     /* accepted nodes, path[0] = 0 */
  uint8_t mask[128];    /* DP run: the skip mask it selected */
  float dp_value;       /* DP run: dp[L][n] */
  double ema[3];        /* DYTC: acceptance estimates after this cycle's update */
} ssd_cycle_record;

/* Copy the log (oldest first) into out[0..max_records-1]; *n_records = entries
 * copied.  The log is cleared by ssd_reset_stats and by switching
 * SSD_OPT_CYCLE_LOG on. */
ssd_status ssd_get_cycle_log(ssd_ctx* ctx, ssd_cycle_record* out, int max_records, int* n_records);

/* Set the DyTC acceptance estimates a_l ([CAS-blog] §3.1) that the next
 * ssd_draft_tree / ssd_generate (DYTC) plans with, e.g. to carry them over
 * from an earlier request.  n_levels in 1..3, every value in [0, 1]. */
ssd_status ssd_set_ema(ssd_ctx* ctx, const double* ema, int n_levels);

/* Generate n_gen tokens after the pending token with the given policy,
 * running the whole draft/verify/accept (and DP refresh) loop inside the
 * library.  out_tokens[0] = the pending token at entry, then the tokens
 * produced, exactly n_gen of them (greedy acceptance makes them identical
 * to plain greedy decoding).  The cache may hold up to draft_k + 1 tokens
 * past the last returned one when generation stops inside a cycle; the
 * committed length and pending token then refer to that state. */
ssd_status ssd_generate(ssd_ctx* ctx, const ssd_policy* policy, int n_gen, int32_t* out_tokens);

/* Latency model of a draft configuration ([CAS-blog] §3.2):
 *   latency_ms = beta[0] + beta[1] * seq_len + beta[2] * layer_depth,
 * layer_depth = layers the pass runs, seq_len = committed context; one model
 * per activation mode (act_int8 0 / 1).
 * ssd_calibrate_latency times one-draft passes with CUDA events on the
 * context's stream (median of reps after one untimed run) over the grid
 * seq_lens[i] x depths[j] (d evenly spaced layers run: layer
 * floor((2m+1) L / 2d), m < d), fits beta by least squares over the points
 * with train[i * n_depths + j] != 0 (train NULL: all), stores it in the
 * context and returns it; times_ms[i * n_depths + j] (may be NULL) receives
 * every point's time.  Needs a prefilled context with 1 <= seq_lens[i] <=
 * committed length; it rolls the committed length back to min(seq_lens)
 * (pending token kept) and overwrites the cache slots past it, like a draft.
 * Errors: INVALID_ARG (ranges, or training points that do not span two
 * sequence lengths and two depths), STATE (no prefill).
 * ssd_set_latency_model stores a given beta (e.g. an earlier calibration).
 * ssd_fit_latency is the least-squares fit alone (host only, no context).
 * ssd_get_level_costs returns the DyTC level costs and the number of levels
 * in use that ssd_generate would plan with now (costs_out[n_levels]). */
ssd_status ssd_calibrate_latency(ssd_ctx* ctx, int act_int8, const int32_t* depths, int n_depths,
                                 const int32_t* seq_lens, int n_seq, int reps, const uint8_t* train, double* beta_out,
                                 double* times_ms);
ssd_status ssd_set_latency_model(ssd_ctx* ctx, int act_int8, const double* beta);
ssd_status ssd_fit_latency(int n, const double* seq_len, const double* depth, const double* ms, double* beta_out);
ssd_status ssd_get_level_costs(ssd_ctx* ctx, const ssd_policy* policy, double* costs_out, int* n_active_out);

/* Cascade depth rules ([CAS-blog] §4.1 item 1, §4.2 problem 3): the largest
 * k <= 3 with 12 * 2^k <= n_layers (= floor(min(3, log2(n_layers / 12)))),
 * one less when seq_len > 512, clamped to [1, n_levels].  Host only. */
int ssd_cascade_depth(int n_layers, int n_levels, int seq_len);

/* The tcgen05 projection's stream-K work split (host side, for checking the
 * division of work without a GPU): `total` (weight tile, K stage) items are
 * cut into G contiguous runs; *begin (may be NULL) = the first item of CTA
 * b's run, *cta (may be NULL) = the CTA whose run holds item i.  Host only. */
void ssd_streamk_split(int64_t total, int G, int b, int64_t i, int64_t* begin, int* cta);
/* The batch-1 GEMV's warp count for a matrix of nu row pairs and `total`
 * (row pair, K chunk) steps, before the grid caps it (host side, as above). */
int64_t ssd_gemv_warps(int nu, int64_t total);
/* The decode attention's key-tile ring rule (host side, as above): for a CTA
 * with `ntile` key tiles, S shared-memory slots and WQ query groups of
 * 16 / WQ warps (WQ in 1..16), *R = the slots in use and *WK = the warp sets
 * sharing the tiles: S and 16 / WQ when no slot is refilled (ntile <= S),
 * else R <= S and WK <= 16 / WQ with R % WK == 0 (every tile of a slot goes
 * to one warp set), the largest such WK and then the largest R.  Either
 * pointer may be NULL.  Invalid arguments write nothing.  Host only. */
void ssd_attn_ring_rule(int ntile, int S, int WQ, int* R, int* WK);

/* sizeof of the ABI's structs, for bindings to check their mirrors: out[0]
 * ssd_model_config, out[1] ssd_policy, out[2] ssd_stats, out[3]
 * ssd_attention_args (n <= 4 entries written).  Host only. */
void ssd_abi_sizes(size_t* out, int n);

/* The host planners alone (no context, no GPU).  ssd_plan_tree: the DyTC
 * tree for acceptance estimates ema[n_levels] and level costs
 * cost[n_levels] (rule stated at SSD_POLICY_DYTC); ssd_plan_hcascade: the
 * horizontal-cascade chain for hc_len[n_levels] (cost, ema, max_nodes,
 * max_depth unused, may be NULL/0).  Outputs: *n_nodes nodes with
 * parents_out[c] (parents_out[0] = -1), and *n_exp expansions in order with
 * exp_node_out[e] and exp_level_out[e].  Arrays must hold 64 entries.
 * Errors: INVALID_ARG (n_levels not in [1, 3], null arrays, max_nodes not in
 * [1, 63], hc_len sum not in [1, 63]). */
ssd_status ssd_plan_tree(int n_levels, const double* ema, const double* cost, int max_nodes, int max_depth,
                         int32_t* parents_out, int* n_nodes, int32_t* exp_node_out, int32_t* exp_level_out,
                         int* n_exp);
ssd_status ssd_plan_hcascade(int n_levels, const int32_t* hc_len, int32_t* parents_out, int* n_nodes,
                             int32_t* exp_node_out, int32_t* exp_level_out, int* n_exp);

/* Plan, draft and return a DyTC tree without verifying it: tokens[0..*n_nodes-1],
 * parents[0..*n_nodes-1] (tokens[0] = pending token, parents[0] = -1).
 * Arrays must hold tree_max_nodes + 1 entries. */
ssd_status ssd_draft_tree(ssd_ctx* ctx, const ssd_policy* policy, int32_t* tokens, int32_t* parents,
                          int* n_nodes);

/* Debug / parity access to the last pass.  ssd_get_logits: fp32 logits of
 * row `row` of the last full-model pass (prefill: the last prompt row is
 * row 0) or draft step.  ssd_get_hidden: fp32 residual after `layer`
 * layers (0 = embedding .. L) of row `row` of the last verify or prefill
 * chunk (the rows whose states the CLaSp target is taken from). */
ssd_status ssd_get_logits(ssd_ctx* ctx, int row, float* out_vocab);
/* Top-1 softmax probabilities of drafts 0..n-1 of the last draft pass that
 * ran with a draft exit threshold (entries past its n_drafted are stale).
 * 1 <= n <= max_rows - 1. */
ssd_status ssd_get_draft_conf(ssd_ctx* ctx, int n, float* out_p1);
ssd_status ssd_get_hidden(ssd_ctx* ctx, int layer, int row, float* out_d);

/* Committed length t and pending token (host copies; no sync). */
ssd_status ssd_get_position(const ssd_ctx* ctx, int32_t* committed_len, int32_t* pending_token);

ssd_status ssd_get_stats(ssd_ctx* ctx, ssd_stats* out);
ssd_status ssd_reset_stats(ssd_ctx* ctx);

/* Implementation switches (for cross-checks and measurement). */
typedef enum {
  SSD_OPT_GEMM_IMPL = 0,  /* 0 = the projections' kernels (register stream-K GEMV for 1 row, tcgen05 for
                             2..64 rows); the only value libssd.so accepts.  The test library
                             libssd_xcheck.so also takes the cross-check kernels: 1 = CUDA-core rows kernel
                             everywhere, 2 = per-row-pair register GEMV for 1 row, 3 = TMA-bulk stream-K
                             GEMV for 1 row; and the tcgen05 work distributions: 4 = split-K in a cluster
                             wherever the tiles fit the SMs, 5 = stream-K everywhere */
  SSD_OPT_USE_GRAPHS = 1, /* 1 (default) = capture decode passes in CUDA graphs, 0 = plain launches */
  SSD_OPT_TIMING = 2,     /* 1 = time every pass with CUDA events (ssd_get_pass_times) */
  SSD_OPT_PDL = 3,        /* 1 (default) = programmatic dependent launch between the kernels of a pass */
  SSD_OPT_L2_PREFETCH_MB = 4, /* MB of the next weight matrix each kernel prefetches into L2 when it ends (default 0 = off) */
  SSD_OPT_TRACE = 5,          /* 1 = record a per-kernel device timeline of each pass (ssd_get_trace) */
  SSD_OPT_CYCLE_LOG = 6       /* 1 = keep the per-cycle log of ssd_generate (ssd_get_cycle_log) */
} ssd_option;
ssd_status ssd_set_option(ssd_ctx* ctx, int option, int value);

/* Per-pass device time in ms, accumulated with CUDA events since the last
 * ssd_reset_stats when timing is enabled (SSD_OPT_TIMING):
 * out[0] draft passes, out[1] verify passes, out[2] DP passes, out[3] AR
 * steps; counts[4] the number of each. */
ssd_status ssd_get_pass_times(ssd_ctx* ctx, double* out_ms, int64_t* counts);

/* Device timeline of the last pass run with SSD_OPT_TRACE on: for each traced
 * kernel i, out[4i] = kind (0 pass set-up, 2 attention, 10 + epilogue of a
 * projection: 10 QKV, 11 residual (W_o or W_d), 12 gate/up, 13 lm_head),
 * out[4i+1] = %globaltimer (ns) when its first CTA became resident,
 * out[4i+2] = when its first CTA passed the dependency wait, out[4i+3] = when
 * its last CTA finished.  *n_entries = kernels written (<= max_entries). */
ssd_status ssd_get_trace(ssd_ctx* ctx, int64_t* out, int max_entries, int* n_entries);

/* Standalone attention over a paged KV cache (one layer), the kernel that the
 * decode passes use.  Row r sees cache slots [0, prefix) and slots base + e
 * for every bit e < rows set in mask[r]: the one visibility rule behind the
 * causal verify, the ancestor mask of tree verification and the per-row
 * mask of CLaSp's batched DP pass that shares the KV cache without copying
 * it ([CLaSp] §三, sequence parallelism; [CAS-paper] abstract, tree).  Each
 * query head h reads KV head h / (n_q_heads / n_kv_heads) (GQA).
 *   q            device fp32 [rows][n_q_heads * head_dim], RoPE applied
 *   k/v_cache    device, element type `dtype` (SSD_BF16, SSD_FP16 or SSD_F32),
 *                [n_layers][n_pages][n_kv_heads][64][head_dim]
 *   block_table  device int32 [n_pages]: logical page -> physical page
 *   out          device fp32 [rows][n_q_heads * head_dim]
 *   q, k/v_cache and out 16-byte aligned.
 * Every slot a row can see must have been written.  A row that sees no
 * slot gets zeros.  Errors: INVALID_ARG (null pointer, unaligned buffer,
 * head_dim not 64/128, n_q_heads not a multiple of n_kv_heads, rows not in
 * 1..64, slot past the block table); CUDA (the launch failed). */
typedef struct {
  const float* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;
  float* out;
  int n_pages, layer, n_q_heads, n_kv_heads, head_dim, dtype;
  int rows, prefix, base;
  uint64_t mask[64];
} ssd_attention_args;

/* Device scratch ssd_attention needs for these shapes: the row descriptor
 * (the key splits merge in distributed shared memory).  0 for shapes that
 * ssd_attention rejects. */
size_t ssd_attention_scratch_bytes(int rows, int n_q_heads, int n_kv_heads, int head_dim);

/* Run the attention on `cuda_stream` using caller-allocated device scratch
 * (256-byte aligned, >= ssd_attention_scratch_bytes).  Asynchronous; the
 * scratch must not be shared by overlapping calls.  The row descriptor is
 * written into the scratch by a kernel launched on the stream (it is passed
 * by value, so no host buffer outlives the call).  A bounded device-side wait
 * that gives up (see SSD_ERR_TIMEOUT) is not reported by this call or by
 * ssd_attention_noalloc: the output is then incomplete. */
ssd_status ssd_attention(const ssd_attention_args* args, void* scratch, size_t scratch_bytes, void* cuda_stream);

/* Allocation-free attention, for callers that may not allocate device
 * memory: code running inside a host framework whose device memory is fully
 * owned by its own pool allocator (a cudaMalloc of its own would fail once the
 * pool has taken the memory, or would fragment it), or on a path that must not
 * call into the allocator at all.  The paper has no counterpart; this is a
 * packaging of ssd_attention.
 * Same arguments, result and errors as ssd_attention; its scratch (the row
 * descriptor, at most 4096 bytes) is one array in device memory that the
 * library reserves statically: every GPU that loads libssd.so holds it until
 * the process exits, and no call allocates anything.  The first call on each
 * device looks up the array's device address (cudaGetSymbolAddress) with that
 * device current; make that first call before any stream capture.  The stream
 * must belong to the current device (INVALID_ARG otherwise).  All calls share
 * the array and each overwrites it: calls that overlap on the GPU (other
 * streams, other threads) race and must be serialised by the caller. */
ssd_status ssd_attention_noalloc(const ssd_attention_args* args, void* cuda_stream);

const char* ssd_last_error(const ssd_ctx* ctx);
const char* ssd_status_string(ssd_status s);
void ssd_destroy(ssd_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif
