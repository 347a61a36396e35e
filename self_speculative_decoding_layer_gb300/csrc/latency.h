// Latency model and cascade-depth rules of the DyTC scheduler (host code).
//
// [CAS-blog] §3.2: each draft configuration's latency is predicted as
//   latency = b0 + b1 * seq_len + b2 * layer_depth
// with the b fitted offline from measurements (the pages report < 15 % error
// on an A100).  layer_depth is read as the number of layers the pass runs and
// seq_len as the committed context it attends over; one model is fitted per
// activation mode (16-bit, int8), since int8 changes the cost per layer.
//
// [CAS-blog] §4.1 item 1: the maximum cascade depth is min(3, log2(layers / 12));
// §4.2 problem 3: one cascade level fewer when seq_len > 512.
#pragma once

namespace ssd {

// Least squares for (b0, b1, b2) over n points (seq_len[i], depth[i]) -> ms[i]:
// the 3x3 normal equations in double, Gaussian elimination with partial
// pivoting.  False (beta untouched) when n < 3 or the points do not determine
// the three coefficients (all seq_len equal, all depths equal, or collinear).
bool fit_latency(int n, const double* seq_len, const double* depth, const double* ms, double beta[3]);

inline double predict_latency(const double beta[3], double seq_len, double depth) {
  return beta[0] + beta[1] * seq_len + beta[2] * depth;
}

// Cascade levels in use: K = floor(min(3, log2(n_layers / 12))) computed
// exactly as the largest k <= 3 with 12 * 2^k <= n_layers, one fewer when
// seq_len > 512, then clamped to [1, n_levels].  The levels kept are the
// first K (the cheapest: L1, then L2).
int cascade_depth(int n_layers, int n_levels, int seq_len);

}  // namespace ssd
