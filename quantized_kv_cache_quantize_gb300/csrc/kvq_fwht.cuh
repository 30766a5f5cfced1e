// Warp-shuffle fast Walsh-Hadamard transform of one row held by a group of
// lanes (8 channels per lane), and BF16 bit helpers.
//
// Rotation (paper section 3, "Hadamard rotation"): x' = (1/sqrt(d)) *
// Sylvester(d) * diag(sigma) * x.  The butterflies run in the order
// h = 1, 2, 4, ..., d/2 (pair (i, i + h) for every i with bit h clear becomes
// (x_i + x_{i+h}, x_i - x_{i+h})), every step a correctly rounded fp32
// operation, then one multiply by fl(1/sqrt(d)).  That order fixes the fp32
// result bit for bit, which is what the quantizer's codes are defined on.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace kvq {

// Lane t of a row group of LPR = d / 8 lanes holds channels 8t .. 8t + 7.
template <int LPR>
__device__ __forceinline__ void fwht_row(float (&x)[8], int t) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if ((e & h) == 0) {
        const float a = x[e], b = x[e + h];
        x[e] = __fadd_rn(a, b);
        x[e + h] = __fsub_rn(a, b);
      }
    }
  }
#pragma unroll
  for (int dl = 1; dl < LPR; dl <<= 1) {
    // lower lane holds x_i: x_i + x_{i+h}; upper lane holds x_{i+h}:
    // x_i - x_{i+h}.  One fused multiply-add with a +-1 factor rounds the
    // exact sum once, exactly like the separate add / subtract.
    const float sgn = (t & dl) ? -1.0f : 1.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float p = __shfl_xor_sync(0xffffffffu, x[e], dl);
      x[e] = __fmaf_rn(sgn, x[e], p);
    }
  }
}

__device__ __forceinline__ uint32_t bf16_bits_rn(float v) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ float bf16_value(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

}  // namespace kvq
