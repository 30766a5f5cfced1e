// Checks the quotient the quantize-append kernels use for a row's (batch,
// head): umulhi(r, m) >> l with (m, l) from kvq::row_divisor, against r / d,
// for every divisor below 5000 on a grid of rows, for random divisors and
// rows below 2^31, and for the last 65536 rows below 2^31 of selected
// divisors.  Prints "checks N bad M"; exits 1 on any mismatch.
#include <cstdint>
#include <cstdio>
#include <random>

#include "../quantized_kv_cache_quantize_gb300/csrc/kvq_internal.h"

int main() {
  std::mt19937_64 rng(1);
  long long bad = 0, checks = 0;
  auto check = [&](uint32_t d, uint32_t r) {
    uint32_t m = 0;
    int sh = 0;
    kvq::row_divisor(d, &m, &sh);
    const uint32_t q = m ? (uint32_t)(((uint64_t)r * m) >> 32) >> sh : (r >> sh);
    ++checks;
    if (q != r / d) {
      if (bad < 5) std::printf("d %u r %u: %u, want %u\n", d, r, q, r / d);
      ++bad;
    }
  };
  for (uint32_t d = 1; d < 5000; ++d)
    for (uint32_t r = 0; r < 20000; r += 7) check(d, r);
  for (int i = 0; i < 1000000; ++i) {
    const uint32_t d = 1 + (uint32_t)(rng() % 0x7FFFFFFFu);
    check(d, (uint32_t)(rng() % 0x80000000u));
    check(d, 0x7FFFFFFFu - (uint32_t)(rng() % 1000));
  }
  for (uint32_t d : {1u, 2u, 3u, 4680u, 6240u, 14400u, 0x40000000u, 0x40000001u, 0x7FFFFFFFu})
    for (uint32_t r = 0x7FFF0000u; r < 0x80000000u; ++r) check(d, r);
  std::printf("checks %lld bad %lld\n", checks, bad);
  return bad == 0 ? 0 : 1;
}
