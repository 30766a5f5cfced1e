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

// rint(fl(x / delta)) (IEEE quotient, ties to even).  q = fl(x * fl(1/delta))
// is within 2^-22 |q| of fl(x / delta), so unless q lies within 2^-20
// max(1, |q|) of a half-integer both round to the same integer; near a
// half-integer (and for non-finite q) the correctly rounded division decides.
__device__ __forceinline__ float rint_div(float x, float delta, float rcp) {
  const float q = __fmul_rn(x, rcp);
  const float n = rintf(q);
  const float margin = __fsub_rn(0.5f, fabsf(__fsub_rn(q, n)));
  if (!(margin > 0x1p-20f * fmaxf(1.0f, fabsf(q)))) return rintf(__fdiv_rn(x, delta));
  return n;
}

template <int D, int BITS, int GROUP>
__global__ void __launch_bounds__(kThreads) quantize_append_kernel(const QuantArgs a) {
  constexpr int LPR = D / 8;                 // lanes per row
  constexpr int RPW = 32 / LPR;              // rows per warp
  constexpr int G = D / GROUP;               // groups per row
  constexpr int LPG = GROUP / 8;             // lanes per group
  constexpr int W = D * BITS / 32;           // 32-bit code words per row
  constexpr int NCH = W / 4;                 // 16-byte code chunks per row
  constexpr int LPC = LPR / NCH;             // lanes per chunk
  constexpr int CODE_BYTES = D * BITS / 8;
  static_assert(NCH >= 1 && LPC >= 1, "layout");
  const float qmax = float((1 << BITS) - 1);

  const int lane = threadIdx.x & 31;
  const int t = lane % LPR;                  // lane within the row group
  const int rbase = lane - t;
  const unsigned per_kv = (unsigned)a.bh * (unsigned)a.n_new;   // < 2^31 (host check)
  const unsigned rows_total = 2u * per_kv;
  const unsigned warp0 = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const unsigned stride = ((gridDim.x * blockDim.x) >> 5) * RPW;
  uint32_t smask[8];
  sign_masks(sign_word_for(a.sign_bits, t), t, smask);

  auto load_row = [&](unsigned r) {
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (r < rows_total) {
      const bool is_v = r >= per_kv;
      const unsigned rk = is_v ? r - per_kv : r;
      raw = __ldg(reinterpret_cast<const uint4*>((is_v ? a.v_new : a.k_new) + (size_t)rk * D + 8 * t));
    }
    return raw;
  };

  unsigned r = warp0 * RPW + lane / LPR;
  uint4 raw = load_row(r);
  for (unsigned r0 = warp0 * RPW; r0 < rows_total; r0 += stride, r += stride) {
    const uint4 next = load_row(r + stride);   // keep the next row's load in flight
    const bool valid = r < rows_total;
    const bool is_v = r >= per_kv;
    const unsigned rk = is_v ? r - per_kv : r;
    const unsigned bh = rk / (unsigned)a.n_new;
    const unsigned tok = rk - bh * (unsigned)a.n_new;

    float x[8];
    load8_masked(raw, smask, x);
    raw = next;
    fwht_row<LPR>(x, t);
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = __fmul_rn(x[e], a.inv_sqrt_d);

    // group min / max (exact operations: order does not matter)
    float mn = fminf(fminf(fminf(x[0], x[1]), fminf(x[2], x[3])), fminf(fminf(x[4], x[5]), fminf(x[6], x[7])));
    float mx = fmaxf(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])), fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7])));
#pragma unroll
    for (int dl = 1; dl < LPG; dl <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, dl));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, dl));
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

    uint32_t word = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float c = __fadd_rn(rint_div(x[e], delta, rcp), zero);
      c = fminf(fmaxf(c, 0.0f), qmax);
      const uint32_t code = (uint32_t)__float2int_rn(c);
      if (BITS == 2) {
        word |= code << (8 * (t & 1) + 2 * (e >> 1) + 16 * (e & 1));
      } else {
        word |= code << (4 * (e >> 1) + 16 * (e & 1));
      }
    }
    if (BITS == 2) word |= __shfl_xor_sync(0xffffffffu, word, 1);

    // 16-byte code chunks: chunk j = words 4j .. 4j+3
    const int j = t / LPC;
    const int wstride = (BITS == 2) ? (LPC / 4) : 1;
    uint4 chunk;
    chunk.x = shfl_idx(word, rbase + LPC * j + 0 * wstride);
    chunk.y = shfl_idx(word, rbase + LPC * j + 1 * wstride);
    chunk.z = shfl_idx(word, rbase + LPC * j + 2 * wstride);
    chunk.w = shfl_idx(word, rbase + LPC * j + 3 * wstride);
    const size_t dst_tok = (size_t)bh * a.cap + a.first + tok;
    if (valid && (t % LPC) == 0) {
      uint8_t* dst = (is_v ? a.v_codes : a.k_codes) + dst_tok * CODE_BYTES + 16 * j;
      *reinterpret_cast<uint4*>(dst) = chunk;
    }

    // (step, zero) record of the token: G words gathered into lane t == 0
    const uint32_t szw = dbits | (zbits << 16);
    uint32_t rec[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int gi = 0; gi < G; ++gi) rec[gi] = shfl_idx(szw, rbase + gi * LPG);
    if (valid && t == 0) {
      uint32_t* dst = (is_v ? a.v_sz : a.k_sz) + dst_tok * G;
      if (G == 4) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(rec[0], rec[1], rec[2], rec[3]);
      } else if (G == 2) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(rec[0], rec[1]);
      } else {
        dst[0] = rec[0];
      }
    }
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
  static int resident = 0;
  if (resident == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &resident, quantize_append_kernel<D, BITS, GROUP>, kThreads, 0) != cudaSuccess ||
        resident < 1)
      resident = 1;
  }
  const long long rows = 2LL * a.bh * a.n_new;
  const int rows_per_block = (kThreads / 32) * (32 / (D / 8));
  long long blocks = (rows + rows_per_block - 1) / rows_per_block;
  const long long cap = (long long)sm_count() * resident;
  if (blocks > cap) blocks = cap;
  quantize_append_kernel<D, BITS, GROUP><<<(unsigned)blocks, kThreads, 0, s>>>(a);
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
