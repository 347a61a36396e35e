// Launch interface of the small kernels in k_misc.cu (internal).
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace ssd {

enum BeginKind { BEGIN_CAUSAL = 0, BEGIN_DRAFT = 1, BEGIN_TREE = 2, BEGIN_EXPAND = 3, BEGIN_DP = 4 };

struct BeginArgs {
  int kind;
  int rows;
  int step;          // DRAFT: draft index k (token = pending if 0, else tok[k-1]); -1: DevState::draft_n
  const int* tok;    // token source
  int tok_offset;    // CAUSAL: first token index in tok
  int first_pending; // CAUSAL: row 0 is the pending token
  const int* depth;  // TREE / EXPAND: node depths
  const unsigned long long* anc;  // TREE / EXPAND: ancestor-or-self bitmask per node
  const int* exp_node;            // EXPAND: node of each expansion
  DevState* st;
  PassDesc* desc;
  const void* E;
  int d;
  int vocab;  // a token id >= vocab (never produced by a correct pass) is embedded as 0 and flagged in DevState::err
  float* h;
  int ldh;
  float* stash0;  // optional: layer-0 stash rows
  int* row_tok;   // optional: token of each row
  unsigned long long* trace;
  // DRAFT with draft exit: the pass's draft length K.  Step 0 opens the gate and
  // marks drafts 0..K-1 invalid (-1) before they are drafted; a later step
  // returns at once when the gate is closed.  0: no draft exit.
  int exit_k;
};

void launch_begin(const BeginArgs& a, int fp16, cudaStream_t st);
// Greedy argmax (ties -> lowest id) and runner-up of `rows` logits rows.  part: argmax_part_bytes(rows)
// of scratch; cnt: rows counters, zero before the launch and left zero after it.
// Draft exit ([CLaSp] experiments: the draft exit threshold).  With st set, the launch is draft `step`
// of an exit-enabled draft pass (one row): it runs only while st->draft_live is 1 (always for step 0),
// also computes the row's top-1 softmax probability p1 = 1 / sum_i exp(x_i - max x) (into
// st->draft_p1[step]), counts the draft (st->draft_n = step + 1) and closes the gate when p1 < thr.
struct ArgmaxExit {
  DevState* st;
  float thr;
  int step;
  // Draft loop in a CUDA graph (a conditional WHILE node around one draft forward): dyn != 0 takes the
  // step from st->draft_n and writes the token to out1[step]; the launch then sets the loop's condition
  // `cond` to 1 while drafting goes on and fewer than k drafts exist.
  int dyn;
  int k;
  int has_cond;
  unsigned long long cond;
};
// Vertical cascade: keep the prefix of drafts[0..k) that am (the higher level's argmax of rows
// pending, drafts[0..k)) agrees with, then its correction, then -1.
void launch_draft_accept(const int* am, int* drafts, int k, cudaStream_t s);
// Before a graph's draft loop: open the gate, draft count 0, drafts 0..k-1 = -1.
void launch_draft_reset(DevState* st, int* drafts, int k, cudaStream_t s);
// Greedy acceptance fused into the verify pass's argmax launch ([CLaSp] §三 stage 2): with st set, the CTA
// that completes the last row's argmax (rows_done counts the rows) runs the acceptance walk over the rows'
// greedy tokens (accept_walk in k_misc.cu), so the verify ends with one launch.
struct AcceptArgs {
  DevState* st;          // null: no acceptance in this launch
  const int* row_tok;    // the verify rows' tokens
  const int* parents;    // null: a chain
  int n_rows;
  int* out_tokens;       // the generation's output buffer, or null
  int* rows_done;        // zero between launches
};
void launch_argmax(const float* logits, int rows, int V, int ld, int* out1, int* out2, void* part, int* cnt,
                   cudaStream_t st, ArgmaxExit ex = ArgmaxExit{}, AcceptArgs acc = AcceptArgs{});
size_t argmax_part_bytes(int rows);
void launch_advance(DevState* st, int rows, const int* am, int take, int* out_tokens, cudaStream_t s);
void launch_compact(const DevState* st, void* kc, void* vc, const int* btab, int n_pages, int n_layers, int n_kv,
                    int hd, int fp16, cudaStream_t s);
void launch_store_children(DevState* st, int* tree_tok, const int* c0, const int* c1, const int* am1, const int* am2,
                           cudaStream_t s);

struct DPStepArgs {
  const DevState* st;
  int i;                 // layer step 1..L
  int lo, hi;            // j range at step i
  int lo_prev, hi_prev;  // j range at step i-1
  const float* h;        // pass rows (layer-i outputs of states (i-1, lo_prev..hi_prev))
  int ldh;
  const float* states_old;  // [ncol, d]
  float* states_new;        // [ncol, d]
  const float* stash_i;     // full-model residual after layer i, rows [stash_rows, d]
  int d;
  float* val;               // [(L+1), ncol]
  unsigned char* back;      // [(L+1), ncol]
  int ncol;
  // The next layer's inputs (null next_h: the last layer): the state chosen for j becomes pass row
  // j - lo of next_h, and, for a tensor-core next layer (next_xb set), its QKV operand rows as 16-bit
  // hi/lo of state * next_gamma ([2][next_mp][d]) and the row's sum of squares next_ss[j - lo] (the RMSNorm
  // hand-off of the residual epilogues, one slot per row).
  float* next_h;
  void* next_xb;
  float* next_ss;
  const void* next_gamma;
  int next_mp;
};

// state(0, 0) = the target's embedding row; it is also the first layer's pass row 0 (h0), with its
// QKV operand rows and sum of squares when xb0 is set (see DPStepArgs::next_xb).
void launch_dp_init(const DevState* st, const float* stash, int d, float* states, float* val, unsigned char* back,
                    float* h0, void* xb0, float* ss0, const void* gamma0, int mp0, int fp16, cudaStream_t s);
void launch_dp_step(const DPStepArgs& a, int fp16, cudaStream_t s);
void launch_dp_backtrack(const unsigned char* back, const float* val, int L, int n, int ncol, unsigned char* mask,
                         float* value, cudaStream_t s);

}  // namespace ssd
