// Eq. (1) of the paper (section 3, "Integer quantization") as the GPU
// quantizers evaluate it: per group the step covering [min, max] and the
// integer zero point, both stored BF16, and every value's code by a
// correctly rounded fp32 quotient, ties to even (IEEE fp32 throughout: no
// fast-math).  Shared by the per-token quantizers (FWHT and tensor-core
// rotation) and the per-channel key quantizer.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "kvq_fwht.cuh"
#include "kvq_sm100.cuh"

namespace kvq {
namespace {

// fl(x / d) from r = fl(1 / d): q0 = fl(x r), the exact residual x - q0 d by
// FMA, one correction step.  Correctly rounded while neither the residual
// nor the quotient leaves the normal range (Markstein's correction with a
// correctly rounded reciprocal).
__device__ __forceinline__ float div_step(float x, float d, float r) {
  const float q0 = __fmul_rn(x, r);
  return __fmaf_rn(__fmaf_rn(-q0, d, x), r, q0);
}

// Eq. (1) for one group given its min and max: the step covering
// [min, max] and the integer zero point, both stored BF16 (the record is
// step | zero << 16), and what the code decision needs.
struct QHdr {
  float delta, rcp, zero;
  int zf;          // the zero point as an integer
  bool fast;       // quotients by the reciprocal and one residual step
  bool clamp;      // some code of the group leaves [0, 2^B - 1]
  uint32_t rec;
};

template <int BITS>
__device__ __forceinline__ QHdr group_header(float mn, float mx) {
  constexpr float qmax = float((1 << BITS) - 1);
  constexpr float kInvQmax = 1.0f / float((1 << BITS) - 1);   // fl(1 / qmax)
  QHdr h;
  const float span = __fsub_rn(mx, mn);
  uint32_t dbits = bf16_bits_rn(span >= 0x1p-100f && span < 0x1p100f
                                    ? div_step(span, qmax, kInvQmax)
                                    : __fdiv_rn(span, qmax));
  if (bf16_value(dbits) == 0.0f) {
    dbits = bf16_bits_rn(fabsf(mn));
    if (bf16_value(dbits) == 0.0f) dbits = 0x3F80u;  // 1.0
  }
  h.delta = bf16_value(dbits);
  h.rcp = __frcp_rn(h.delta);
  h.fast = h.rcp < 0x1p100f && fabsf(mn) * h.rcp < 0x1p21f && fabsf(mx) * h.rcp < 0x1p21f;
  const float zq = h.fast ? div_step(-mn, h.delta, h.rcp) : __fdiv_rn(-mn, h.delta);
  const uint32_t zbits = bf16_bits_rn(__fadd_rn(rintf(zq), 0.0f));
  h.zero = bf16_value(zbits);
  h.zf = __float2int_rn(h.zero);
  h.rec = dbits | (zbits << 16);
  // codes are monotone in x: those of the group's min and max bound them all
  const float kMagic = 12582912.0f;   // 1.5 * 2^23
  auto code_of = [&](float v) {
    const float q0 = __fmul_rn(v, h.rcp);
    const float q = __fmaf_rn(__fmaf_rn(-q0, h.delta, v), h.rcp, q0);
    return __fadd_rn(__fadd_rn(q, kMagic), h.zero) - kMagic;
  };
  h.clamp = h.fast && (code_of(mn) < 0.0f || code_of(mx) > qmax);
  return h;
}

// The code of one value of a group with header h (the arithmetic of
// group_codes below, one value at a time).
template <int BITS>
__device__ __forceinline__ uint32_t code_of_value(float v, const QHdr& h) {
  constexpr float qmax = float((1 << BITS) - 1);
  const float kMagic = 12582912.0f;   // 1.5 * 2^23
  if (h.fast) {
    const float q0 = __fmul_rn(v, h.rcp);
    const float q = __fmaf_rn(__fmaf_rn(-q0, h.delta, v), h.rcp, q0);
    const float t = __fadd_rn(q, kMagic);
    if (h.clamp) return __float_as_uint(fminf(fmaxf(__fadd_rn(t, h.zero), kMagic), kMagic + qmax)) - 0x4B400000u;
    return (uint32_t)((int)(__float_as_uint(t) - 0x4B400000u) + h.zf);
  }
  const float t = fminf(fmaxf(__fadd_rn(rintf(__fdiv_rn(v, h.delta)), h.zero), 0.0f), qmax);
  return (uint32_t)__float2int_rn(t);
}

// Eq. (1) for one group (or the part of it one thread holds) given the
// group's min and max; the n values xg[0..n) are replaced by
// 1.5 * 2^23 + code - zfold, zfold being the zero point when it is left for
// the packing to add (0 otherwise).  Returns the record (step | zero << 16).
//
// Fast route: q = fl(x / delta) exactly, from the correctly rounded
// reciprocal r and one residual step (q0 = fl(x r), e = x - q0 delta exact
// by FMA, q = fl(q0 + e r): correctly rounded while nothing over- or
// underflows); rint(q) by adding 1.5 * 2^23 (ties to even, |q| < 2^21); the
// integer zero point added after the rounding.  K = 1.5 * 2^23 + code then
// carries the code in its low mantissa bits.  The clamp to [0, 2^B - 1] is
// needed only when the code of the group's min or max falls outside; when
// it is not, the zero point is left to the packing (which adds it to a whole
// half-word of codes at once).
//
// apply_codes does the per-value part for n values of a group whose header
// is h (a group may be coded in parts: every part takes the same zfold).
template <int BITS, int N>
__device__ __forceinline__ void apply_codes(float* xg, const QHdr& h, int& zfold) {
  const float qmax = float((1 << BITS) - 1);
  const float kMagic = 12582912.0f;   // 1.5 * 2^23
  if (h.fast) {
    const uint64_t r2 = ptx::f2_pack(h.rcp, h.rcp);
    const uint64_t nd2 = ptx::f2_pack(-h.delta, -h.delta);
    const uint64_t m2 = ptx::f2_pack(kMagic, kMagic);
#pragma unroll
    for (int c = 0; c < N; c += 2) {
      const uint64_t xv = ptx::f2_pack(xg[c], xg[c + 1]);
      const uint64_t q0 = ptx::f2_mul(xv, r2);
      const uint64_t e = ptx::f2_fma(q0, nd2, xv);
      const uint64_t q = ptx::f2_fma(e, r2, q0);
      ptx::f2_unpack(ptx::f2_add(q, m2), xg[c], xg[c + 1]);
    }
    zfold = h.zf;
    if (h.clamp) {
#pragma unroll
      for (int c = 0; c < N; ++c) xg[c] = fminf(fmaxf(__fadd_rn(xg[c], h.zero), kMagic), kMagic + qmax);
      zfold = 0;
    }
  } else {
    zfold = 0;
    // exact division element by element (huge quotients, tiny steps): a rare
    // path, kept as one rolled loop over a local copy so that its divisions
    // do not sit unrolled in the kernel's hot code
    float tmp[N];
#pragma unroll
    for (int c = 0; c < N; ++c) tmp[c] = xg[c];
#pragma unroll 1
    for (int c = 0; c < N; ++c) {
      float t = __fadd_rn(rintf(__fdiv_rn(tmp[c], h.delta)), h.zero);
      t = fminf(fmaxf(t, 0.0f), qmax);
      tmp[c] = __fadd_rn(t, kMagic);
    }
#pragma unroll
    for (int c = 0; c < N; ++c) xg[c] = tmp[c];
  }
}

template <int BITS, int N>
__device__ __forceinline__ uint32_t group_codes(float* xg, float mn, float mx, int& zfold) {
  const QHdr h = group_header<BITS>(mn, mx);
  apply_codes<BITS, N>(xg, h, zfold);
  return h.rec;
}

// One packed word from the 32/BITS consecutive channels xw[0..) (each value
// 1.5 * 2^23 + code): channel 2k + h of the word at bits BITS*k + 16h.  The
// low 16 bits of 1.5 * 2^23 are zero, so a Horner sum of the bit patterns
// (times 2^BITS per code) leaves the codes in the low half-word, given the
// group's folded zero point (all channels of a word share one group).
template <int BITS>
__device__ __forceinline__ uint32_t pack_word(const float* xw, int zfold) {
  constexpr int PER_WORD = 32 / BITS;
  // zfold times (1 + 2^BITS + 2^(2 BITS) + ...) over a half-word's codes
  constexpr uint32_t kOnes = BITS == 2 ? 0x5555u : 0x1111u;
  uint32_t half[2];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    uint32_t acc = __float_as_uint(xw[hh + 2 * (PER_WORD / 2 - 1)]);
#pragma unroll
    for (int k = PER_WORD / 2 - 2; k >= 0; --k) acc = acc * (1u << BITS) + __float_as_uint(xw[hh + 2 * k]);
    half[hh] = acc + (uint32_t)zfold * kOnes;
  }
  return __byte_perm(half[0], half[1], 0x5410);
}

// min and max of n values (two new values per 3-input min / max)
template <int N>
__device__ __forceinline__ void min_max(const float* v, float& mn, float& mx) {
  mn = v[0];
  mx = v[0];
#pragma unroll
  for (int c = 1; c < N; c += 2) {
    const float u = v[c], w = c + 1 < N ? v[c + 1] : u;
    mn = fminf(mn, fminf(u, w));
    mx = fmaxf(mx, fmaxf(u, w));
  }
}

}  // namespace
}  // namespace kvq
