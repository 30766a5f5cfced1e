/* Checks the identity the quantizer's code path relies on: for a divisor d
 * and r = fl(1/d) (correctly rounded), q0 = fl(x r), e = fma(-q0, d, x) and
 * q = fma(e, r, q0) give q = fl(x / d), the correctly rounded quotient
 * (Markstein's correction step), while nothing over- or underflows.
 * Divisors: every normal BF16 value with exponent in [lo, hi); numerators:
 * `per` pseudo-random floats of magnitude ~2^-4 .. 2^4 times the divisor,
 * plus every exact half-integer quotient (k + 1/2) d for |k| <= 8.
 * Prints "checked N mismatches M" and exits 1 on any mismatch. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

static int check(float x, float d, float r) {
  const float q0 = x * r;
  const float e = fmaf(-q0, d, x);
  const float q = fmaf(e, r, q0);
  const float ref = x / d;
  return to_bits(q) == to_bits(ref);
}

int main(int argc, char** argv) {
  const int lo = argc > 1 ? atoi(argv[1]) : -20, hi = argc > 2 ? atoi(argv[2]) : 13;
  const int per = argc > 3 ? atoi(argv[3]) : 2000;
  uint32_t seed = 12345u;
  unsigned long long n = 0, bad = 0;
  for (int ex = lo; ex < hi; ++ex) {
    for (uint32_t m = 0; m < 128; ++m) {
      const uint32_t e = (uint32_t)(127 + ex);
      const float d = from_bits((e << 23) | (m << 16));
      const float r = 1.0f / d;
      for (int i = 0; i < per; ++i) {
        seed = seed * 1664525u + 1013904223u;
        const uint32_t xe = e - 4 + (seed >> 29);
        seed = seed * 1664525u + 1013904223u;
        float x = from_bits((xe << 23) | (seed >> 9));
        if (seed & 256u) x = -x;
        ++n;
        if (!check(x, d, r)) ++bad;
      }
      for (int k = -8; k <= 8; ++k) {
        const float x = ((float)k + 0.5f) * d;
        ++n;
        if (!check(x, d, r)) ++bad;
      }
    }
  }
  printf("checked %llu mismatches %llu\n", n, bad);
  return bad != 0;
}
