// Code tables for the kernels, built on the host from their definitions:
// NF4 (the QLoRA data type) and, for comparison, the 4-bit float E2M1.
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
#include <cstring>
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

// The 16 levels of a code table, fp32, ascending.
void levels(int quant_type, float (&out)[16]) {
  if (quant_type == QL_FP4) {
    // E2M1: magnitude m * 0.5 for exponent 0 (subnormal), 2^(e-1) (1 + m / 2)
    // otherwise; the 8 magnitudes, negated and not, scaled by 1 / 6
    double mags[8];
    for (int e = 0, i = 0; e < 4; ++e)
      for (int m = 0; m < 2; ++m, ++i) mags[i] = e == 0 ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
    int n = 0;
    for (int i = 7; i >= 1; --i) out[n++] = (float)(-mags[i] / mags[7]);
    for (int i = 0; i < 8; ++i) out[n++] = (float)(mags[i] / mags[7]);
    out[15] = 1.0f;  // 15 distinct values; the last index repeats +1
    return;
  }
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
  for (int i = 0; i < 16; ++i) out[i] = (float)lv[i];
  out[0] = -1.0f;
  out[15] = 1.0f;
  out[7] = 0.0f;
}

Codebook build(int quant_type) {
  Codebook cb{};
  levels(quant_type, cb.q);

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
      std::fprintf(stderr, "libqlora: coding cell %d holds %d thresholds\n", c, inside);
      std::abort();
    }
    cb.cell_lo[c] = below;
    cb.cell_u[c] = uin;
    double delta = 0x1p-30;
    if (std::isfinite(uin)) {
      const double tb = 0.5 * ((double)std::nextafterf(uin, -INFINITY) + (double)uin);  // exact
      delta = (double)uin - tb;
    }
    uint32_t db;
    const float df = (float)delta;
    std::memcpy(&db, &df, 4);
    if ((db & 0x7FFFFFu) != 0 || !(df > 0.0f)) {
      std::fprintf(stderr, "libqlora: cell %d: rounding step %g not a normal power of two\n", c, delta);
      std::abort();
    }
    cb.cell_d[c] = db | (uint32_t)(below + 1);
  }
  // One-FMA test: is there a quotient W / Mi * 2^k (W, Mi in [128, 255], the
  // significands of normal bf16 values; quotients near a threshold of
  // magnitude >= 2^-6 never involve a subnormal w) in [t', u) for some u?
  cb.one_fma = true;
  for (int j = 0; j < 15 && cb.one_fma; ++j) {
    const double uu = std::fabs((double)u[j]);
    const double tb = std::fabs(0.5 * ((double)std::nextafterf(u[j], -INFINITY) + (double)u[j]));
    const double lo = std::fmin(uu, tb), hi = std::fmax(uu, tb);
    for (int W = 128; W < 256 && cb.one_fma; ++W)
      for (int Mi = 128; Mi < 256 && cb.one_fma; ++Mi) {
        const double rho = (double)W / (double)Mi;
        const int k = (int)std::floor(std::log2(hi / rho));
        for (int kk = k - 1; kk <= k + 1; ++kk) {
          const double qv = std::ldexp(rho, kk);  // within 2^-50 of the exact ratio: the window is 2^-25 wide
          if (qv >= lo - 0x1p-40 * hi && qv <= hi + 0x1p-40 * hi) cb.one_fma = false;
        }
      }
  }
  // The quantizer picks the cell from an approximate quotient (relative error
  // below 2^-21); a threshold that close to a cell boundary could then be
  // skipped.  None is: every threshold keeps at least 2^-16 from every boundary.
  for (int j = 0; j < 15; ++j)
    for (int c = 0; c <= kCells; ++c) {
      const double b = (c - 32.5) / 32.0;
      if (std::fabs((double)u[j] - b) < 0x1p-16) {
        std::fprintf(stderr, "libqlora: threshold %d lies within 2^-16 of a coding-cell boundary\n", j);
        std::abort();
      }
    }
  return cb;
}

}  // namespace

const Codebook &codebook(int quant_type) {
  static Codebook cb[2];
  static std::once_flag once[2];
  const int t = quant_type == QL_FP4 ? 1 : 0;
  std::call_once(once[t], [t] { cb[t] = build(t == 1 ? QL_FP4 : QL_NF4); });
  return cb[t];
}

}  // namespace ql

extern "C" int ql_codebook(int32_t quant_type, float *out16) {
  if (!out16) return ql::set_error(QL_ERR_INVALID, "ql_codebook: null output");
  if (quant_type != QL_NF4 && quant_type != QL_FP4)
    return ql::set_error(QL_ERR_UNSUPPORTED, "ql_codebook: quant type %d (0 = NF4, 1 = FP4)", quant_type);
  const ql::Codebook &cb = ql::codebook(quant_type);
  for (int i = 0; i < 16; ++i) out16[i] = cb.q[i];
  return QL_OK;
}

extern "C" int ql_nf4_codebook(float *out16) { return ql_codebook(QL_NF4, out16); }
