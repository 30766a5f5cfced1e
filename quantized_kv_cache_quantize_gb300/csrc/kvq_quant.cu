// The rotation kernel (sm_103a): the attention's operands (the query as FP16
// high and low parts, the current chunk's values as FP16) and its range
// check.  It rotates with the fast Walsh-Hadamard transform (paper section
// 3, "Hadamard rotation"): fp32 butterflies in the order h = 1, 2, ..., d/2,
// then one multiply by fl(1/sqrt(d)), every step a correctly rounded fp32
// operation, so the result is fixed bit for bit.  The quantize-append
// (per token and group, and the per-channel keys) rotates on the tensor
// cores: kvq_quant_mma.cu.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kvq_checks.cuh"
#include "kvq_eq1.cuh"
#include "kvq_fwht.cuh"
#include "kvq_internal.h"
#include "kvq_sm100.cuh"

namespace kvq {

namespace {


// sign word of lane t's channels without indexing a kernel-parameter array at
// run time (which would copy the parameters to local memory)
__device__ __forceinline__ uint32_t sign_word_for(const uint32_t (&sb)[4], int t) {
  const int i = (8 * t) >> 5;
  return i == 0 ? sb[0] : i == 1 ? sb[1] : i == 2 ? sb[2] : sb[3];
}

// Rotation of Q and V_R to FP16 (with the FP16 remainder when asked).
// LPR = d / 32 lanes per row, 32 channels per
// lane: lane j first holds channels [32j, 32j + 32) and runs the butterflies
// h = 1 .. 16 in registers; one transpose through shared memory then gives
// it channels {32u + (32 / LPR) j + v} (u < LPR, v < 32 / LPR), whose
// butterflies h = 32 (and 64) are again in registers.  Same fp32 operations
// in the same order as the textbook transform (h = 1, 2, ..., d/2, then the
// multiply by fl(1/sqrt(d))), so the FP16 outputs are the oracle's fp32
// rotation rounded.  Each lane's next row is loaded before the current one
// is transformed.
constexpr int kRotThreads = 256;
constexpr int kRotBlocksPerSm = 2;

template <int D>
__global__ void __launch_bounds__(kRotThreads, kRotBlocksPerSm) rotate_kernel(const RotateArgs a) {
  constexpr int LPR = D / 32;          // lanes per row
  constexpr int RPW = 32 / LPR;        // rows per warp
  constexpr int VW = 32 / LPR;         // contiguous channels per lane after the transpose
  __shared__ __align__(16) float tbuf[kRotThreads / 32][RPW][D];
  const int lane = threadIdx.x & 31;
  const int j = lane % LPR;            // channel block of the lane
  const int g = lane / LPR;            // row within the warp's rows
  float* rowbuf = tbuf[threadIdx.x >> 5][g];
  const long long total = a.rows[0] + a.rows[1];
  const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long step = (((long long)gridDim.x * blockDim.x) >> 5) * RPW;

  // the lane's 32 sign bits regrouped: bit k = channel 2k, bit 16 + k =
  // channel 2k + 1, so that (z << (15 - k)) & 0x80008000 is the sign mask of
  // the 32-bit word holding channels 2k (low half) and 2k + 1 (high half)
  const uint32_t sw = sign_word_for(a.sign_bits, 4 * j);
  uint32_t z = 0;
#pragma unroll
  for (int k = 0; k < 16; ++k) z |= (((sw >> (2 * k)) & 1u) << k) | (((sw >> (2 * k + 1)) & 1u) << (16 + k));
  const long long rows0 = a.rows[0];
  const uint16_t* src0 = a.src[0];
  const uint16_t* src1 = a.src[1];

  auto load = [&](long long r, uint4 (&raw)[4]) {
    if (r < total) {
      const bool s1 = r >= rows0;
      const uint16_t* srcp = (s1 ? src1 : src0) + (s1 ? r - rows0 : r) * D + 32 * j;
#pragma unroll
      for (int k = 0; k < 4; ++k) raw[k] = __ldg(reinterpret_cast<const uint4*>(srcp) + k);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) raw[k] = make_uint4(0u, 0u, 0u, 0u);
    }
  };

  bool out_of_range = false;
  long long r = warp0 * RPW + g;
  uint4 nxt[4];
  load(r, nxt);
  // the loop bounds are warp-uniform (r - g steps by whole warps)
  for (; r - g < total; r += step) {
    uint4 raw[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) raw[k] = nxt[k];
    load(r + step, nxt);

    float x[32];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t t = w[i] ^ ((z << (15 - (4 * k + i))) & 0x80008000u);
        const float lo = __uint_as_float(t << 16), hi = __uint_as_float(t & 0xFFFF0000u);
        x[8 * k + 2 * i] = __fadd_rn(lo, hi);       // h = 1
        x[8 * k + 2 * i + 1] = __fsub_rn(lo, hi);
      }
    }
#pragma unroll
    for (int h = 2; h < 32; h <<= 1) {
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        if ((i & h) == 0) {
          const uint64_t A = ptx::f2_pack(x[i], x[i + 1]);
          const uint64_t B = ptx::f2_pack(x[i + h], x[i + h + 1]);
          ptx::f2_unpack(ptx::f2_add(A, B), x[i], x[i + 1]);
          ptx::f2_unpack(ptx::f2_sub(A, B), x[i + h], x[i + h + 1]);
        }
      }
    }
    // transpose through the row's buffer.  Chunk c (4 floats) of the
    // channels of lane jj sits at float 32 jj + 4 (c ^ sw(jj)), sw(jj) =
    // (32 / LPR) / 4 * jj + (g mod 8 / LPR): the eight lanes of a quarter-warp
    // meet eight different bank groups on both the writes and the reads
    auto swz = [&](int jj) { return (VW / 4) * jj + (g & (8 / LPR - 1)); };
    __syncwarp();
    {
      const int sj = swz(j);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4*>(rowbuf + 32 * j + 4 * (c ^ sj)) =
            make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]);
    }
    __syncwarp();
    // read: y[VW u + v] = channel 32u + VW j + v
    float y[32];
#pragma unroll
    for (int u = 0; u < LPR; ++u) {
      const int su = swz(u);
#pragma unroll
      for (int w4 = 0; w4 < VW / 4; ++w4) {
        const float4 v = *reinterpret_cast<const float4*>(rowbuf + 32 * u + 4 * (((VW / 4) * j + w4) ^ su));
        y[VW * u + 4 * w4] = v.x; y[VW * u + 4 * w4 + 1] = v.y;
        y[VW * u + 4 * w4 + 2] = v.z; y[VW * u + 4 * w4 + 3] = v.w;
      }
    }
    // h = 32 (and 64): pairs (u, u + h/32) at the same v
#pragma unroll
    for (int hu = 1; hu < LPR; hu <<= 1) {
#pragma unroll
      for (int u = 0; u < LPR; ++u) {
        if ((u & hu) == 0) {
#pragma unroll
          for (int v = 0; v < VW; v += 2) {
            const uint64_t A = ptx::f2_pack(y[VW * u + v], y[VW * u + v + 1]);
            const uint64_t B = ptx::f2_pack(y[VW * (u + hu) + v], y[VW * (u + hu) + v + 1]);
            ptx::f2_unpack(ptx::f2_add(A, B), y[VW * u + v], y[VW * u + v + 1]);
            ptx::f2_unpack(ptx::f2_sub(A, B), y[VW * (u + hu) + v], y[VW * (u + hu) + v + 1]);
          }
        }
      }
    }
    {
      const uint64_t s2 = ptx::f2_pack(a.inv_sqrt_d, a.inv_sqrt_d);
#pragma unroll
      for (int i = 0; i < 32; i += 2) ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(y[i], y[i + 1]), s2), y[i], y[i + 1]);
    }
    if (r >= total) continue;
    const bool s1 = r >= rows0;
    const long long rr = s1 ? r - rows0 : r;
    if (!KVQ_IN_BOUNDS(rr, s1 ? a.rows[1] : a.rows[0], a.status, a.bounds_site)) continue;
    void* dstp = s1 ? a.dst[1] : a.dst[0];
    uint16_t* lop = s1 ? a.dst_lo[1] : a.dst_lo[0];
    const float lim = s1 ? a.range_limit[1] : a.range_limit[0];
    if (lim > 0.f) {
      // largest magnitude, NaN propagated (a NaN is out of range too)
      float mx = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) asm("max.NaN.f32 %0, %0, %1;" : "+f"(mx) : "f"(fabsf(y[i])));
      out_of_range |= !(mx < lim);
    }
#pragma unroll
    for (int u = 0; u < LPR; ++u) {
      const long long off = rr * D + 32 * u + VW * j;   // first channel of this run
      {
        uint32_t hw[VW / 2], lw[VW / 2];
#pragma unroll
        for (int q2 = 0; q2 < VW / 2; ++q2) {
          const float e0 = y[VW * u + 2 * q2], e1 = y[VW * u + 2 * q2 + 1];
          hw[q2] = ptx::f16x2_rn(e0, e1);
          const float b0 = __half2float(__ushort_as_half((unsigned short)(hw[q2] & 0xFFFFu)));
          const float b1 = __half2float(__ushort_as_half((unsigned short)(hw[q2] >> 16)));
          lw[q2] = ptx::f16x2_rn(__fsub_rn(e0, b0), __fsub_rn(e1, b1));
        }
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(dstp) + off);
#pragma unroll
        for (int q8 = 0; q8 < VW / 8; ++q8)
          dst[q8] = make_uint4(hw[4 * q8], hw[4 * q8 + 1], hw[4 * q8 + 2], hw[4 * q8 + 3]);
        if (lop != nullptr) {
          uint4* dl = reinterpret_cast<uint4*>(lop + off);
#pragma unroll
          for (int q8 = 0; q8 < VW / 8; ++q8)
            dl[q8] = make_uint4(lw[4 * q8], lw[4 * q8 + 1], lw[4 * q8 + 2], lw[4 * q8 + 3]);
        }
      }
    }
  }
  // a rotated value the FP16 operands cannot carry: recorded, not fatal
  // (the loop bounds are warp-uniform, so every lane arrives here)
  if (__any_sync(0xffffffffu, out_of_range) && lane == 0 && a.status != nullptr)
    atomicCAS(a.status, 0, (int)KVQ_ERR_RANGE);
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

long long grid_for_rows(long long rows, int rows_per_block, int blocks_per_sm) {
  long long blocks = (rows + rows_per_block - 1) / rows_per_block;
  const long long cap = (long long)sm_count() * blocks_per_sm;   // one resident wave
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return blocks;
}

}  // namespace

cudaError_t launch_rotate(const RotateArgs& a, int d, cudaStream_t stream) {
  const long long rows = a.rows[0] + a.rows[1];
  if (rows == 0) return cudaSuccess;
  const int rows_per_block = (kRotThreads / 32) * (32 / (d / 32));
  const unsigned grid = (unsigned)grid_for_rows(rows, rows_per_block, kRotBlocksPerSm);
  if (d == 64) {
    rotate_kernel<64><<<grid, kRotThreads, 0, stream>>>(a);
    note_launch();
  } else {
    rotate_kernel<128><<<grid, kRotThreads, 0, stream>>>(a);
    note_launch();
  }
  return cudaGetLastError();
}

}  // namespace kvq
