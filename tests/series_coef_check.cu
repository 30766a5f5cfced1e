// Prints the polynomial of log(sinh a / a) that the exact-correction kernels
// use (constexpr functions of the attention kernel header): the number of
// terms, the range of a^2 it covers and its coefficients (sinhc_fit), one
// value per line, for the CPU test that checks them.
#include <cstdio>

#include "../quantized_kv_cache_quantize_gb300/csrc/kvq_attn_kernel.cuh"

int main() {
  std::printf("%d\n%.9e\n", kvq::kFitTerms, (double)kvq::kFitTmax);
  for (int k = 0; k < kvq::kFitTerms; ++k) std::printf("%.9e\n", (double)kvq::sinhc_fit(k));
  return 0;
}
