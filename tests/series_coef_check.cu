// Prints the series coefficients of log(sinh a / a) that the exact-correction
// kernels use (sinhc_coef, a host-and-device constexpr of the attention
// kernel header) and the number of terms, one per line, for the CPU test
// that checks them against the Bernoulli-number formula.
#include <cstdio>

#include "../quantized_kv_cache_quantize_gb300/csrc/kvq_attn_kernel.cuh"

int main() {
  std::printf("%d\n", kvq::kSeriesTerms);
  for (int k = 0; k < kvq::kSeriesTerms; ++k) std::printf("%.9e\n", (double)kvq::sinhc_coef(k));
  return 0;
}
