// Quantize-append and rotation kernels (sm_103a).
//
// Quantize-append: for every new K and V row, rotate (randomized Hadamard,
// paper section 3), quantize per token and group with Eq. (1) (asymmetric
// round-to-nearest, step and zero point covering [min, max]) and pack the
// codes into the chunk slot of the sliding-window cache.
//
// Mapping: a row of d channels is held by d/8 consecutive lanes, 8 channels
// (one 16-byte load) per lane; a warp holds 32/(d/8) rows.  The transform,
// the group min/max and the packing all move data with warp shuffles; codes
// leave in 16-byte stores, the (step, zero) record of a token in one store.
// The kernel is bound by HBM bandwidth: per row it reads 2d bytes and writes
// d*bits/8 + 4*(d/group) bytes.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kvq_fwht.cuh"
#include "kvq_internal.h"
#include "kvq_sm100.cuh"

namespace kvq {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t shfl_idx(uint32_t v, int src) {
  return __shfl_sync(0xffffffffu, v, src);
}

__device__ __forceinline__ uint32_t h_bits_rn(float v) {
  return (uint32_t)__half_as_ushort(__float2half_rn(v));
}

// sign word of lane t's channels without indexing a kernel-parameter array at
// run time (which would copy the parameters to local memory)
__device__ __forceinline__ uint32_t sign_word_for(const uint32_t (&sb)[4], int t) {
  const int i = (8 * t) >> 5;
  return i == 0 ? sb[0] : i == 1 ? sb[1] : i == 2 ? sb[2] : sb[3];
}

// Sign flips of the randomized rotation in the BF16 pair domain: word i of
// a row holds channels 2i (low half) and 2i + 1 (high half); XOR with m[i]
// flips their sign bits (bit 15, bit 31).
struct PairSigns {
  uint32_t m[64];
};

constexpr int kRowThreads = 128;

// One thread per row (one token's K or V row of one head): the whole row in
// registers, so the rotation needs no data exchange between threads.  Per
// row: d/8 16-byte loads, fp32 butterflies in the order h = 1, 2, ..., d/2
// (packed fp32 pairs from h = 2 on: each lane is the same correctly rounded
// add or subtract), per-group min/max, Eq. (1) codes, packed 16-byte stores.
template <int D, int BITS, int GROUP>
__global__ void __launch_bounds__(kRowThreads) quantize_rows_kernel(const QuantArgs a,
                                                                    const PairSigns sg) {
  constexpr int G = D / GROUP;
  constexpr int CODE_BYTES = D * BITS / 8;
  constexpr int PER_WORD = 32 / BITS;
  const float qmax = float((1 << BITS) - 1);

  const unsigned per_kv = (unsigned)a.bh * (unsigned)a.n_new;   // < 2^31 (host check)
  const unsigned r = blockIdx.x * kRowThreads + threadIdx.x;
  if (r >= 2u * per_kv) return;
  const bool is_v = r >= per_kv;
  const unsigned rk = is_v ? r - per_kv : r;
  const unsigned bh = rk / (unsigned)a.n_new;
  const unsigned tok = rk - bh * (unsigned)a.n_new;

  const uint4* src = reinterpret_cast<const uint4*>((is_v ? a.v_new : a.k_new) + (size_t)rk * D);
  float x[D];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) {
    const uint4 raw = __ldg(src + i);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t ws = w[k] ^ sg.m[4 * i + k];
      x[8 * i + 2 * k] = __uint_as_float(ws << 16);
      x[8 * i + 2 * k + 1] = __uint_as_float(ws & 0xFFFF0000u);
    }
  }
  // butterflies: h = 1 on scalars, then packed pairs (x_i, x_i+1)
#pragma unroll
  for (int i = 0; i < D; i += 2) {
    const float u = x[i], v = x[i + 1];
    x[i] = __fadd_rn(u, v);
    x[i + 1] = __fsub_rn(u, v);
  }
#pragma unroll
  for (int h = 2; h < D; h <<= 1) {
#pragma unroll
    for (int i = 0; i < D; i += 2) {
      if ((i & h) == 0) {
        const uint64_t A = ptx::f2_pack(x[i], x[i + 1]);
        const uint64_t B = ptx::f2_pack(x[i + h], x[i + h + 1]);
        ptx::f2_unpack(ptx::f2_add(A, B), x[i], x[i + 1]);
        ptx::f2_unpack(ptx::f2_sub(A, B), x[i + h], x[i + h + 1]);
      }
    }
  }
  {
    const uint64_t s2 = ptx::f2_pack(a.inv_sqrt_d, a.inv_sqrt_d);
#pragma unroll
    for (int i = 0; i < D; i += 2) ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(x[i], x[i + 1]), s2), x[i], x[i + 1]);
  }

  uint32_t rec[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float mn = x[GROUP * g], mx = x[GROUP * g];
#pragma unroll
    for (int c = 1; c < GROUP; c += 2) {
      const float u = x[GROUP * g + c], v = c + 1 < GROUP ? x[GROUP * g + c + 1] : u;
      mn = fminf(mn, fminf(u, v));
      mx = fmaxf(mx, fmaxf(u, v));
    }
    // Eq. (1): step covering [min, max], integer zero point, both stored BF16
    uint32_t dbits = bf16_bits_rn(__fdiv_rn(__fsub_rn(mx, mn), qmax));
    if (bf16_value(dbits) == 0.0f) {
      dbits = bf16_bits_rn(fabsf(mn));
      if (bf16_value(dbits) == 0.0f) dbits = 0x3F80u;  // 1.0
    }
    const float delta = bf16_value(dbits);
    const float rcp = __frcp_rn(delta);
    const uint32_t zbits = bf16_bits_rn(__fadd_rn(rintf(__fdiv_rn(-mn, delta)), 0.0f));
    const float zero = bf16_value(zbits);
    rec[g] = dbits | (zbits << 16);

    // codes.  Fast route: q = fl(x / delta) exactly, from the correctly
    // rounded reciprocal r and one residual step (q0 = fl(x r), e = x - q0 delta
    // exact by FMA, q = fl(q0 + e r): correctly rounded while nothing over- or
    // underflows); rint(q) by adding 1.5 * 2^23 (ties to even, |q| < 2^21);
    // the integer zero point added after the rounding.  K = 1.5 * 2^23 + code
    // then carries the code in its low mantissa bits.  Codes are monotone in
    // x, so those of the group's min and max bound them all and the clamp to
    // [0, 2^B - 1] is needed only when one of those two falls outside.
    const float kMagic = 12582912.0f;   // 1.5 * 2^23
    const bool fast = rcp < 0x1p100f && fabsf(mn) * rcp < 0x1p21f && fabsf(mx) * rcp < 0x1p21f;
    float* xg = x + GROUP * g;
    if (fast) {
      auto code_of = [&](float v) {
        const float q0 = __fmul_rn(v, rcp);
        const float q = __fmaf_rn(__fmaf_rn(-q0, delta, v), rcp, q0);
        return __fadd_rn(__fadd_rn(q, kMagic), zero) - kMagic;
      };
      const bool clamp = code_of(mn) < 0.0f || code_of(mx) > qmax;
      const uint64_t r2 = ptx::f2_pack(rcp, rcp);
      const uint64_t nd2 = ptx::f2_pack(-delta, -delta);
      const uint64_t m2 = ptx::f2_pack(kMagic, kMagic);
      const uint64_t z2 = ptx::f2_pack(zero, zero);
#pragma unroll
      for (int c = 0; c < GROUP; c += 2) {
        const uint64_t xv = ptx::f2_pack(xg[c], xg[c + 1]);
        const uint64_t q0 = ptx::f2_mul(xv, r2);
        const uint64_t e = ptx::f2_fma(q0, nd2, xv);
        const uint64_t q = ptx::f2_fma(e, r2, q0);
        ptx::f2_unpack(ptx::f2_add(ptx::f2_add(q, m2), z2), xg[c], xg[c + 1]);
      }
      if (clamp) {
#pragma unroll
        for (int c = 0; c < GROUP; ++c) xg[c] = fminf(fmaxf(xg[c], kMagic), kMagic + qmax);
      }
    } else {
      // exact division element by element (huge quotients, tiny steps)
#pragma unroll
      for (int c = 0; c < GROUP; ++c) {
        float t = __fadd_rn(rintf(__fdiv_rn(xg[c], delta)), zero);
        t = fminf(fmaxf(t, 0.0f), qmax);
        xg[c] = __fadd_rn(t, kMagic);
      }
    }
  }

  // pack: channel ch = 16w + 2k + h (INT2) / 8w + 2k + h (INT4) -> bits
  // BITS*k + 16h.  The low 16 bits of 1.5 * 2^23 are zero, so a Horner sum
  // of the K bit patterns (times 2^BITS per code) leaves exactly the codes
  // in the low half-word.
  uint32_t words[D * BITS / 32];
#pragma unroll
  for (int w = 0; w < D * BITS / 32; ++w) {
    uint32_t half[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      uint32_t acc = __float_as_uint(x[PER_WORD * w + hh + 2 * (PER_WORD / 2 - 1)]);
#pragma unroll
      for (int k = PER_WORD / 2 - 2; k >= 0; --k)
        acc = acc * (1u << BITS) + __float_as_uint(x[PER_WORD * w + hh + 2 * k]);
      half[hh] = acc;
    }
    words[w] = __byte_perm(half[0], half[1], 0x5410);
  }

  const size_t dst_tok = (size_t)bh * a.cap + a.first + tok;
  uint4* dc = reinterpret_cast<uint4*>((is_v ? a.v_codes : a.k_codes) + dst_tok * CODE_BYTES);
#pragma unroll
  for (int i = 0; i < CODE_BYTES / 16; ++i)
    dc[i] = make_uint4(words[4 * i], words[4 * i + 1], words[4 * i + 2], words[4 * i + 3]);
  uint32_t* ds = (is_v ? a.v_sz : a.k_sz) + dst_tok * G;
  if (G == 4) {
    *reinterpret_cast<uint4*>(ds) = make_uint4(rec[0], rec[1 % G], rec[2 % G], rec[3 % G]);
  } else if (G == 2) {
    *reinterpret_cast<uint2*>(ds) = make_uint2(rec[0], rec[1 % G]);
  } else {
    ds[0] = rec[0];
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads) rotate_kernel(const RotateArgs a) {
  constexpr int LPR = D / 8;
  constexpr int RPW = 32 / LPR;
  const int lane = threadIdx.x & 31;
  const int t = lane % LPR;
  const long long total = a.rows[0] + a.rows[1];
  const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const uint32_t sign_word = sign_word_for(a.sign_bits, t);

  for (long long r0 = warp0 * RPW; r0 < total; r0 += nwarps * RPW) {
    const long long r = r0 + lane / LPR;
    const bool valid = r < total;
    long long rr = valid ? r : 0;
    const bool seg1 = rr >= a.rows[0];
    if (seg1) rr -= a.rows[0];
    const uint16_t* srcp = seg1 ? a.src[1] : a.src[0];
    void* dstp = seg1 ? a.dst[1] : a.dst[0];
    uint16_t* lop = seg1 ? a.dst_lo[1] : a.dst_lo[0];
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (valid) raw = __ldg(reinterpret_cast<const uint4*>(srcp + rr * D + 8 * t));
    float x[8];
    load8_signed(raw, sign_word, t, x);
    fwht_row<LPR>(x, t);
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = __fmul_rn(x[e], a.inv_sqrt_d);
    if (!valid) continue;
    if (a.out_f32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(dstp) + rr * D + 8 * t);
      dst[0] = make_float4(x[0], x[1], x[2], x[3]);
      dst[1] = make_float4(x[4], x[5], x[6], x[7]);
    } else {
      uint32_t hb[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) hb[e] = h_bits_rn(x[e]);
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(dstp) + rr * D + 8 * t) =
          make_uint4(hb[0] | (hb[1] << 16), hb[2] | (hb[3] << 16), hb[4] | (hb[5] << 16),
                     hb[6] | (hb[7] << 16));
      if (lop != nullptr) {
        uint32_t lb[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          lb[e] = h_bits_rn(__fsub_rn(x[e], __half2float(__ushort_as_half((unsigned short)hb[e]))));
        *reinterpret_cast<uint4*>(lop + rr * D + 8 * t) =
            make_uint4(lb[0] | (lb[1] << 16), lb[2] | (lb[3] << 16), lb[4] | (lb[5] << 16),
                       lb[6] | (lb[7] << 16));
      }
    }
  }
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      n = 148;
    }
  }
  return n;
}

long long grid_for_rows(long long rows, int rows_per_block) {
  long long blocks = (rows + rows_per_block - 1) / rows_per_block;
  const long long cap = (long long)sm_count() * 8;  // 8 blocks of 256 threads per SM
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return blocks;
}

template <int D, int BITS, int GROUP>
cudaError_t launch_q(const QuantArgs& a, cudaStream_t s) {
  PairSigns sg;
  for (int i = 0; i < 64; ++i) {
    const int c0 = 2 * i, c1 = 2 * i + 1;
    const uint32_t s0 = c0 < D ? (a.sign_bits[c0 >> 5] >> (c0 & 31)) & 1u : 0u;
    const uint32_t s1 = c1 < D ? (a.sign_bits[c1 >> 5] >> (c1 & 31)) & 1u : 0u;
    sg.m[i] = (s0 << 15) | (s1 << 31);
  }
  const long long rows = 2LL * a.bh * a.n_new;
  const unsigned blocks = (unsigned)((rows + kRowThreads - 1) / kRowThreads);
  quantize_rows_kernel<D, BITS, GROUP><<<blocks, kRowThreads, 0, s>>>(a, sg);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize_append(const QuantArgs& a, int d, int bits, int group,
                                   cudaStream_t stream, bool* supported) {
  *supported = true;
#define KVQ_Q(D_, B_, G_) \
  if (d == D_ && bits == B_ && group == G_) return launch_q<D_, B_, G_>(a, stream);
  KVQ_Q(64, 2, 32)
  KVQ_Q(64, 2, 64)
  KVQ_Q(64, 4, 32)
  KVQ_Q(64, 4, 64)
  KVQ_Q(128, 2, 32)
  KVQ_Q(128, 2, 64)
  KVQ_Q(128, 4, 32)
  KVQ_Q(128, 4, 64)
#undef KVQ_Q
  *supported = false;
  return cudaSuccess;
}

cudaError_t launch_rotate(const RotateArgs& a, int d, cudaStream_t stream) {
  const long long rows = a.rows[0] + a.rows[1];
  if (rows == 0) return cudaSuccess;
  const int rows_per_block = (kThreads / 32) * (32 / (d / 8));
  const unsigned grid = (unsigned)grid_for_rows(rows, rows_per_block);
  if (d == 64) {
    rotate_kernel<64><<<grid, kThreads, 0, stream>>>(a);
  } else {
    rotate_kernel<128><<<grid, kThreads, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace kvq
