// NF4 codebook for the kernels, built on the host from its definition.
//
// NF4 ("4-bit NormalFloat", QLoRA abstract, innovation (a); news write-up: the
// data type that is information-theoretically optimal for normally distributed
// weights) has 16 levels that are standard-normal quantiles normalised to
// [-1, 1] with an exact zero.  With both endpoints and a zero among 16 levels
// the grid is asymmetric: 8 positive levels are the quantiles at 8
// probabilities equally spaced from DELTA towards 1/2, 7 negative levels the
// negated quantiles at 7 probabilities equally spaced from DELTA towards 1/2,
// plus 0; all divided by the quantile at DELTA, DELTA = 1 - (1/32 + 1/30)/2.
// Levels are built in double and rounded once to float.
//
// The standard-normal quantile is found by bisection on the CDF
// Phi(x) = erfc(-x / sqrt 2) / 2 until the bracket cannot shrink further.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "common.cuh"

namespace ql {
namespace {

double normal_cdf(double x) { return 0.5 * std::erfc(-x / std::sqrt(2.0)); }

double normal_quantile(double p) {
  double lo = -40.0, hi = 40.0;
  for (int it = 0; it < 2000; ++it) {
    double mid = 0.5 * (lo + hi);
    if (mid <= lo || mid >= hi) break;
    if (normal_cdf(mid) < p) lo = mid; else hi = mid;
  }
  return 0.5 * (lo + hi);
}

Codebook build() {
  Codebook cb{};
  const double delta = 1.0 - 0.5 * (1.0 / 32.0 + 1.0 / 30.0);
  const double zmax = normal_quantile(delta);
  double lv[16];
  int n = 0;
  // negative side: 7 probabilities delta - i (delta - 1/2) / 7, i = 0..6, most negative first
  for (int i = 0; i < 7; ++i) {
    double p = delta - i * ((delta - 0.5) / 7.0);
    lv[n++] = -normal_quantile(p) / zmax;
  }
  lv[n++] = 0.0;
  // positive side: 8 probabilities delta - i (delta - 1/2) / 8, i = 7..0, ascending
  for (int i = 7; i >= 0; --i) {
    double p = delta - i * ((delta - 0.5) / 8.0);
    lv[n++] = normal_quantile(p) / zmax;
  }
  for (int i = 0; i < 16; ++i) cb.q[i] = (float)lv[i];
  cb.q[0] = -1.0f;
  cb.q[15] = 1.0f;
  cb.q[7] = 0.0f;

  // Decision thresholds: t_j = (q_j + q_{j+1}) / 2 (exact in double).  An fp32
  // x lies above t_j exactly when x >= u_j, the smallest float above t_j.
  float u[15];
  for (int j = 0; j < 15; ++j) {
    double t = 0.5 * ((double)cb.q[j] + (double)cb.q[j + 1]);
    float f = (float)t;
    if ((double)f <= t) f = std::nextafterf(f, INFINITY);
    u[j] = f;
  }
  // Cells: x maps to c = rne(32x + 32), so cell c holds x in
  // [(c - 32.5)/32, (c - 31.5)/32] (both ends, for ties).
  for (int c = 0; c < kCells; ++c) {
    double lo = (c - 32.5) / 32.0, hi = (c - 31.5) / 32.0;
    int below = 0, inside = 0;
    float uin = INFINITY;
    for (int j = 0; j < 15; ++j) {
      if ((double)u[j] <= lo) ++below;
      else if ((double)u[j] <= hi) { ++inside; uin = u[j]; }
    }
    if (inside > 1) {
      std::fprintf(stderr, "libqlora: NF4 coding cell %d holds %d thresholds\n", c, inside);
      std::abort();
    }
    cb.cell_lo[c] = below;
    cb.cell_u[c] = uin;
  }
  return cb;
}

}  // namespace

const Codebook &codebook() {
  static Codebook cb;
  static std::once_flag once;
  std::call_once(once, [] { cb = build(); });
  return cb;
}

}  // namespace ql

extern "C" int ql_nf4_codebook(float *out16) {
  if (!out16) return ql::set_error(QL_ERR_INVALID, "ql_nf4_codebook: null output");
  const ql::Codebook &cb = ql::codebook();
  for (int i = 0; i < 16; ++i) out16[i] = cb.q[i];
  return QL_OK;
}
