// Latency model fit and cascade-depth rule (definitions in latency.h).
#include "latency.h"

#include <math.h>

namespace ssd {

bool fit_latency(int n, const double* s, const double* d, const double* y, double beta[3]) {
  if (n < 3) return false;
  // normal equations A^T A b = A^T y with rows (1, s_i, d_i)
  double M[3][4] = {};
  for (int i = 0; i < n; ++i) {
    const double r[3] = {1.0, s[i], d[i]};
    for (int a = 0; a < 3; ++a) {
      for (int b = 0; b < 3; ++b) M[a][b] += r[a] * r[b];
      M[a][3] += r[a] * y[i];
    }
  }
  double scale = 0.0;  // singularity test relative to the matrix's size
  for (int a = 0; a < 3; ++a)
    for (int b = 0; b < 3; ++b) scale = fmax(scale, fabs(M[a][b]));
  for (int c = 0; c < 3; ++c) {
    int piv = c;
    for (int r = c + 1; r < 3; ++r)
      if (fabs(M[r][c]) > fabs(M[piv][c])) piv = r;
    if (!(fabs(M[piv][c]) > 1e-12 * scale)) return false;
    if (piv != c)
      for (int k = 0; k < 4; ++k) {
        const double t = M[c][k];
        M[c][k] = M[piv][k];
        M[piv][k] = t;
      }
    for (int r = c + 1; r < 3; ++r) {
      const double f = M[r][c] / M[c][c];
      for (int k = c; k < 4; ++k) M[r][k] -= f * M[c][k];
    }
  }
  double b[3];
  for (int c = 2; c >= 0; --c) {
    double v = M[c][3];
    for (int k = c + 1; k < 3; ++k) v -= M[c][k] * b[k];
    b[c] = v / M[c][c];
  }
  for (int c = 0; c < 3; ++c) beta[c] = b[c];
  return true;
}

int cascade_depth(int n_layers, int n_levels, int seq_len) {
  int k = 0;  // floor(log2(n_layers / 12)) capped at 3; below 12 layers the bound is under 1
  while (k < 3 && 12LL * (2LL << k) <= n_layers) ++k;
  if (12 > n_layers) k = 0;
  if (seq_len > 512) k -= 1;
  if (k > n_levels) k = n_levels;
  return k < 1 ? 1 : k;
}

}  // namespace ssd
