/* Exhaustive check of the quantizer's division-free quotient.
 *
 * For every pair of bf16 values w, m with |w| <= m and m in [2^-60, 2^60]
 * (the range where the kernel uses it), compares
 *   r = RN(1/m); x0 = RN(w r); x = RN(x0 + RN(w - x0 m) r)   (FMA steps)
 * with the IEEE quotient RN(w / m).  They must agree whenever either is at
 * least 2^-12 in magnitude; below that every value codes to the NF4 zero
 * level, whose nearest decision thresholds are beyond 0.039 in magnitude.
 * Exit status 0 and "bad 0" on success. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float from_bits(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }

int main(void) {
  long long bad = 0, tested = 0;
  for (uint32_t mb = 1; mb < 0x7F80; ++mb) {
    float m = from_bits(mb << 16);
    if (!(m >= 0x1p-60f && m <= 0x1p60f)) continue;
    float r = 1.0f / m;
    for (uint32_t wb = 0; wb <= mb; ++wb) {
      for (int s = 0; s < 2; ++s) {
        float w = from_bits((wb << 16) | (s ? 0x80000000u : 0u));
        float x0 = w * r;
        float res = fmaf(-x0, m, w);
        float x = fmaf(res, r, x0);
        float ref = w / m;
        ++tested;
        if (x != ref && (fabsf(ref) >= 0x1p-12f || fabsf(x) >= 0x1p-12f)) {
          if (bad < 5) printf("mismatch w=%a m=%a x=%a ref=%a\n", w, m, x, ref);
          ++bad;
        }
      }
    }
  }
  printf("tested %lld bad %lld\n", tested, bad);
  return bad != 0;
}
