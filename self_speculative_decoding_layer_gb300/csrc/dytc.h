// DyTC (dynamic tree cascade) routing on the host: acceptance-rate EMA per
// cascade level and latency-aware tree construction.
//
// [CAS-blog] §3.1: a_l <- alpha * rate_l + (1 - alpha) * a_l, alpha = 0.2;
// §4.1 item 2: start near 0.6-0.7 (0.65 here).  §3.2: latency is predicted
// as b0 + b1 * seq_len + b2 * layer_depth; at batch 1 a pass costs the bytes
// of the layers it runs plus the lm_head, so c_l = that over a full pass.
// [CAS-paper] abstract: DyTC routes the multi-level drafts and assigns the
// draft lengths from acceptance-rate and latency heuristics.  The pages give
// no exact rule; the one implemented (identically in the CPU oracle):
//   root p = 1; expanding node u at level l adds a rank-0 child with
//   p(u) a_l and a rank-1 child with p(u) (1 - a_l) a_l;
//   E = 1 + sum p(non-root), T = 1 + sum c over expansions;
//   candidates: unexpanded nodes with depth < max_depth, levels <= the
//   level that created the node (root: any), so each child's layers were run
//   for all of its ancestors (nested skip sets);
//   gain = p a + p (1 - a) a; best gain / c (ties: lower node, then lower
//   level); expand while gain / c > E / T and a node slot is free; the
//   rank-1 child needs a free slot too.
// All arithmetic is IEEE double in the written order; this file is compiled
// without multiply-add contraction so plans match the oracle exactly.
#pragma once

#include <vector>

namespace ssd {

struct TreePlan {
  std::vector<int> parents, depth, cap;
  std::vector<double> prob;
  std::vector<int> exp_node, exp_level, child0, child1;  // per expansion; child id 0 = absent
};

TreePlan dytc_plan(const std::vector<double>& a, const std::vector<double>& c, int max_nodes, int max_depth);

// Horizontal cascade ([CAS-paper] abstract names vertical and horizontal cascades as the classic
// baselines DyTC improves on; the horizontal one drafts the earlier positions of a chain with the more
// accurate levels and the later ones with the cheaper levels): a chain of sum(lens) drafts, the first
// lens[n_levels-1] by the highest level, then lens[n_levels-2] by the next, ..., the last lens[0] by L1.
// Nested levels make every layer a later (cheaper) draft runs already written for the earlier drafts.
TreePlan hcascade_plan(const int* lens, int n_levels);

// One EMA step: every expanded node on the accepted walk path[0..n_acc] is an
// event of its level, a success when the target argmax at that node equals
// the token of its rank-0 child.
void dytc_update(std::vector<double>& a, double alpha, const TreePlan& plan, const int* tokens, const int* argmax,
                 const int* path, int n_acc);

}  // namespace ssd
