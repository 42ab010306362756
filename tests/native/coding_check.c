/* Exhaustive check of the quantizer's division-free coding.
 *
 * Input (argv[1..16]): the 16 fp32 codebook levels, ascending, as hex floats.
 * For every pair of bf16 values w, m with |w| <= m and m in [2^-60, 2^60]
 * (the kernel's fast path), compares
 *   reference: code = #{ j : RN(w / m) >= u_j }, u_j the smallest float above
 *              the exact midpoint t_j = (q_j + q_{j+1}) / 2 (IEEE division);
 *   method:    cell = low byte of RN(32 w r + 1.5 * 2^23 + 32) with r within
 *              two ulps of 1/m (every r from RN(1/m) - 2 ulp to + 2 ulp is
 *              tried), then from the cell's row (u, delta | lower + 1):
 *              e = fma(-m, u, w), v = fma(m, delta', e),
 *              code = (lower + 1) - [v < 0];
 *   one-FMA:   the same with v = e, which the library uses when no quotient of
 *              two normal bf16 values lies between t' = u - delta and u (it
 *              decides that by enumerating significand pairs, as done here).
 * The two-FMA method must match everywhere; the one-FMA method must match
 * whenever the enumeration allows it ("one_fma 1").
 * The table is built as the library builds it: cells of width 1/32 over
 * [-1, 1] (cell c holds x with rne(32 x + 32) = c), at most one threshold per
 * cell, delta = u - (pred(u) + u) / 2, rows past cell 64 without threshold.
 * Also checks every threshold keeps 2^-16 from every cell boundary.
 * Exit status 0 and "bad 0" on success. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float from_bits(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }
static uint32_t to_bits(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }

static float cell_u[256];
static uint32_t cell_d[256];
static float uth[15];

static int ref_code(float x) {
  int c = 0;
  for (int j = 0; j < 15; ++j) c += x >= uth[j];
  return c;
}

static int method_code(float w, float m, float r, int one_fma) {
  const float r32 = r * 32.0f;
  const uint32_t cell = to_bits(fmaf(w, r32, 12582944.0f)) & 0xFFu;
  const float e = fmaf(-m, cell_u[cell], w);
  const float v = one_fma ? e : fmaf(m, from_bits(cell_d[cell]), e);
  return (int)(cell_d[cell] & 31u) + ((to_bits(v) >> 31) ? -1 : 0);
}

/* No quotient W / Mi * 2^k of normal bf16 significands in the window between
 * t' and u of any threshold (then one FMA decides). */
static int one_fma_allowed(void) {
  for (int j = 0; j < 15; ++j) {
    const double uu = fabs((double)uth[j]);
    const double tb = fabs(0.5 * ((double)nextafterf(uth[j], -INFINITY) + (double)uth[j]));
    const double lo = fmin(uu, tb), hi = fmax(uu, tb);
    for (int W = 128; W < 256; ++W)
      for (int Mi = 128; Mi < 256; ++Mi) {
        const double rho = (double)W / (double)Mi;
        const int k = (int)floor(log2(hi / rho));
        for (int kk = k - 1; kk <= k + 1; ++kk) {
          const double qv = ldexp(rho, kk);
          if (qv >= lo - 0x1p-40 * hi && qv <= hi + 0x1p-40 * hi) return 0;
        }
      }
  }
  return 1;
}

int main(int argc, char **argv) {
  if (argc != 17) {
    fprintf(stderr, "usage: coding_check q0 ... q15\n");
    return 2;
  }
  float q[16];
  for (int i = 0; i < 16; ++i) q[i] = strtof(argv[i + 1], NULL);
  for (int j = 0; j < 15; ++j) {
    double t = 0.5 * ((double)q[j] + (double)q[j + 1]);
    float f = (float)t;
    if ((double)f <= t) f = nextafterf(f, INFINITY);
    uth[j] = f;
  }
  for (int c = 0; c < 256; ++c) {
    cell_u[c] = INFINITY;
    cell_d[c] = 0x30800000u | 8u;
  }
  for (int c = 0; c <= 64; ++c) {
    double lo = (c - 32.5) / 32.0, hi = (c - 31.5) / 32.0;
    int below = 0, inside = 0;
    float uin = INFINITY;
    for (int j = 0; j < 15; ++j) {
      if ((double)uth[j] <= lo) ++below;
      else if ((double)uth[j] <= hi) { ++inside; uin = uth[j]; }
    }
    if (inside > 1) { printf("cell %d holds %d thresholds\n", c, inside); return 1; }
    double delta = 0x1p-30;
    if (isfinite(uin)) delta = (double)uin - 0.5 * ((double)nextafterf(uin, -INFINITY) + (double)uin);
    cell_u[c] = uin;
    cell_d[c] = to_bits((float)delta) | (uint32_t)(below + 1);
  }
  for (int j = 0; j < 15; ++j)
    for (int c = 0; c <= 65; ++c)
      if (fabs((double)uth[j] - (c - 32.5) / 32.0) < 0x1p-16) {
        printf("threshold %d near boundary %d\n", j, c);
        return 1;
      }
  const int one_fma = one_fma_allowed();
  long long bad = 0, bad1 = 0, tested = 0;
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : bad, bad1, tested)
  for (uint32_t mb = 1; mb < 0x7F80; ++mb) {
    const float m = from_bits(mb << 16);
    if (!(m >= 0x1p-60f && m <= 0x1p60f)) continue;
    const float r0 = 1.0f / m;
    float rs[5];
    rs[2] = r0;
    rs[1] = nextafterf(r0, 0.0f);
    rs[0] = nextafterf(rs[1], 0.0f);
    rs[3] = nextafterf(r0, INFINITY);
    rs[4] = nextafterf(rs[3], INFINITY);
    for (uint32_t wb = 0; wb <= mb; ++wb) {
      for (int s = 0; s < 2; ++s) {
        const float w = from_bits((wb << 16) | (s ? 0x80000000u : 0u));
        const int ref = ref_code(w / m);
        for (int k = 0; k < 5; ++k) {
          ++tested;
          const int got = method_code(w, m, rs[k], 0);
          if (got != ref) {
#pragma omp critical
            if (bad < 5) printf("mismatch w=%a m=%a r=%a code %d ref %d\n", w, m, rs[k], got, ref);
            ++bad;
          }
          if (method_code(w, m, rs[k], 1) != ref) ++bad1;
        }
      }
    }
  }
  printf("one_fma %d one-FMA mismatches %lld\n", one_fma, bad1);
  if (one_fma && bad1) bad += bad1;
  printf("tested %lld bad %lld\n", tested, bad);
  return bad != 0;
}
