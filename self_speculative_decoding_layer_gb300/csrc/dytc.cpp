// DyTC host policy (rule stated in dytc.h).
#include "dytc.h"

namespace ssd {

TreePlan dytc_plan(const std::vector<double>& a, const std::vector<double>& c, int max_nodes, int max_depth) {
  TreePlan p;
  const int nl = (int)a.size();
  std::vector<char> expanded;
  p.parents.push_back(-1);
  p.depth.push_back(0);
  p.prob.push_back(1.0);
  p.cap.push_back(nl - 1);
  expanded.push_back(0);
  double E = 1.0, T = 1.0;
  while (true) {
    bool have = false;
    double best = 0.0;
    int bu = -1, bl = -1;
    for (int u = 0; u < (int)p.parents.size(); ++u) {
      if (expanded[u] || p.depth[u] >= max_depth) continue;
      for (int l = 0; l <= p.cap[u]; ++l) {
        const double al = a[l];
        const double gain = p.prob[u] * al + p.prob[u] * (1.0 - al) * al;
        const double score = gain / c[l];
        if (!have || score > best) {
          have = true;
          best = score;
          bu = u;
          bl = l;
        }
      }
    }
    if (!have || (int)p.parents.size() - 1 >= max_nodes || !(best > E / T)) break;
    const double al = a[bl];
    expanded[bu] = 1;
    p.exp_node.push_back(bu);
    p.exp_level.push_back(bl);
    const double probs[2] = {p.prob[bu] * al, p.prob[bu] * (1.0 - al) * al};
    int kids[2] = {0, 0};
    for (int r = 0; r < 2; ++r) {
      if ((int)p.parents.size() - 1 >= max_nodes) break;
      kids[r] = (int)p.parents.size();
      p.parents.push_back(bu);
      p.depth.push_back(p.depth[bu] + 1);
      p.prob.push_back(probs[r]);
      p.cap.push_back(bl);
      expanded.push_back(0);
      E += probs[r];
    }
    p.child0.push_back(kids[0]);
    p.child1.push_back(kids[1]);
    T += c[bl];
  }
  return p;
}

TreePlan hcascade_plan(const int* lens, int n_levels) {
  TreePlan p;
  p.parents.push_back(-1);
  p.depth.push_back(0);
  p.prob.push_back(1.0);
  p.cap.push_back(n_levels - 1);
  int r = 0;
  for (int l = n_levels - 1; l >= 0; --l)
    for (int i = 0; i < lens[l]; ++i, ++r) {
      p.exp_node.push_back(r);
      p.exp_level.push_back(l);
      p.child0.push_back(r + 1);
      p.child1.push_back(0);
      p.parents.push_back(r);
      p.depth.push_back(r + 1);
      p.prob.push_back(1.0);
      p.cap.push_back(l);
    }
  return p;
}

void dytc_update(std::vector<double>& a, double alpha, const TreePlan& plan, const int* tokens, const int* argmax,
                 const int* path, int n_acc) {
  const int nl = (int)a.size();
  std::vector<int> ev(nl, 0), ok(nl, 0);
  for (int i = 0; i <= n_acc; ++i) {
    const int u = path[i];
    for (size_t e = 0; e < plan.exp_node.size(); ++e) {
      if (plan.exp_node[e] != u) continue;
      const int l = plan.exp_level[e];
      ev[l] += 1;
      if (plan.child0[e] > 0 && argmax[u] == tokens[plan.child0[e]]) ok[l] += 1;
    }
  }
  for (int l = 0; l < nl; ++l)
    if (ev[l]) a[l] = alpha * ((double)ok[l] / (double)ev[l]) + (1.0 - alpha) * a[l];
}

}  // namespace ssd
