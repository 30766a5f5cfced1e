// Fused Jensen-bias-corrected chunk attention over a low-bit KV window
// (sm_103a: TMA, tcgen05 MMA into tensor memory).
//
// Paper: "Quantized Keys Steal Attention" -- abstract and section 1 (the
// current chunk attends over the cached window and itself; a per-score
// correction b, from the cached keys' step sizes and the query norm, is
// subtracted before the softmax from cached-key scores only), Figure 3
// caption (b removes the Jensen bias E[exp(s + delta)] > exp(s)), section 3
// (Eq. (1) dequantization, Hadamard rotation), Figure 2 caption (the masses
// P_S and P_R).
//
// One CTA of 128 threads owns 128 query rows of one (batch, head); thread r
// owns row r (TMEM lane r).  Per 128-key tile:
//   cached tile : every thread dequantizes one key's packed K and V row into
//                 FP16 tiles in shared memory (128-byte swizzle), plus the
//                 bias columns of that key;
//   current tile: TMA loads the ORIGINAL BF16 keys and the rotated FP16
//                 values;
//   S           : tcgen05 MMAs (M 128, N 128, K 16 steps) into TMEM.  Cached
//                 tiles: Q' K_hat'^T in FP16 (plus Q'_lo K_hat'^T with the
//                 precise-query flag), then one K=16 MMA adds
//                 -(scale/24) sum_g n_jg D_ig^2 through 16 extra columns (bias
//                 folded into the contraction).  Current tiles: Q K^T on the
//                 unrotated BF16 inputs (exact products);
//   softmax     : online, one shared running max, two running sums (cached,
//                 current); P to shared memory as FP16;
//   O += P V    : tcgen05 MMAs into TMEM (V operand MN-major).
// Epilogue: O / (l_S + l_R), inverse rotation per row (FWHT in registers),
// BF16 store; P_S = l_S / (l_S + l_R), P_R = l_R / (l_S + l_R).
//
// Operand precision: cached-segment operands are FP16 (11 significant bits,
// the same MMA rate as BF16).  INT2 dequantized values (code - z) * D with a
// BF16 step D need at most 10 significant bits, so the cached K/V tiles are
// exact; the rotated query carries one FP16 rounding unless it is split into
// high and low parts.  Current-segment scores use the BF16 inputs as they
// are.  Requires |values| < 65504 after rotation (FP16 range).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kvq_internal.h"
#include "kvq_sm100.cuh"

namespace kvq {

namespace {

__device__ int g_attn_status;

struct AttnParams {
  const uint8_t* k_codes;
  const uint8_t* v_codes;
  const uint32_t* k_sz;
  const uint32_t* v_sz;
  int n_s, cap, n_q, n_r;
  float scale_log2;   // scale * log2(e)
  float alpha_coef;   // -(scale / 24) with the correction, 0 without
  int corr;
  int precise_query;
  int mass_only;
  uint16_t* out;
  float* p_s;
  float* p_r;
  uint32_t sign_bits[4];
  float inv_sqrt_d;
  unsigned long long wait_limit_ns;
};

constexpr int kThreads = 128;
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
constexpr int kHalf = 16384;  // one [128 rows][64 x 16-bit] swizzled sub-tile

template <int D>
struct Smem {
  static constexpr int kTile = kBlockM * D * 2;
  static constexpr int kQ = 0;                       // rotated queries, FP16 (high part)
  static constexpr int kQlo = kQ + kTile;            // FP16 low part
  static constexpr int kQo = kQlo + kTile;           // original queries, BF16
  static constexpr int kK = kQo + kTile;
  static constexpr int kV = kK + kTile;
  static constexpr int kP = kV + kTile;              // 128 x 128 fp16
  static constexpr int kQx = kP + 2 * kHalf;         // 2 x [128 x 16] fp16, no swizzle
  static constexpr int kKx = kQx + 8192;
  static constexpr int kBar = kKx + 8192;
  static constexpr int kBytes = kBar + 64;
  static constexpr int kAlloc = kBytes + 1024;       // slack for 1024-byte alignment
};

// Wait for an mbarrier phase with a time limit; false (and the status word
// set) when the limit ran out.
__device__ bool wait_bounded(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > limit_ns) {
      atomicCAS(&g_attn_status, 0, (int)KVQ_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// byte offset of 16-byte chunk `c` (0..7) of row `r` in a 128-byte-swizzled
// [rows][64 x 16-bit] sub-tile
__device__ __forceinline__ int sw128(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

// byte offset of element (row, k) of a [128][16] 16-bit K-major tile without
// swizzle: 8-row x 16-byte core matrices, K chunks 128 B apart, row groups 256 B
__device__ __forceinline__ int noswz16(int r, int kchunk) {
  return (r >> 3) * 256 + kchunk * 128 + (r & 7) * 16;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float h_lo(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu))); }
__device__ __forceinline__ float h_hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Dequantize one packed row (codes + per-group (step, zero) words) into an
// FP16 row of the swizzled tile at `tile` (row r).  WITH_ZERO: x_hat =
// (code - z) * D (Eq. (1)); without: code * D only, which is exact in FP16
// for INT2 (<= 10 significant bits) -- the zero-point term of the keys is
// added through the extension columns instead.  Writes D/8 16-byte chunks.
template <int D, int BITS, int GROUP, bool WITH_ZERO>
__device__ __forceinline__ void dequant_row(const uint32_t* words, const uint32_t* sz,
                                            uint8_t* tile, int r) {
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {
    const int g = (8 * c) / GROUP;
    const float delta = bf16_lo(sz[g]);
    const float zero = WITH_ZERO ? bf16_hi(sz[g]) : 0.0f;
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t c0, c1;
      if (BITS == 2) {
        const uint32_t w = words[c >> 1];
        const int k = 4 * (c & 1) + i;
        c0 = (w >> (2 * k)) & 3u;
        c1 = (w >> (2 * k + 16)) & 3u;
      } else {
        const uint32_t w = words[c];
        c0 = (w >> (4 * i)) & 15u;
        c1 = (w >> (4 * i + 16)) & 15u;
      }
      const float v0 = __fmul_rn(__fsub_rn((float)c0, zero), delta);
      const float v1 = __fmul_rn(__fsub_rn((float)c1, zero), delta);
      out[i] = pack_h2(v0, v1);
    }
    const int half = c >> 3;
    *reinterpret_cast<uint4*>(tile + half * kHalf + sw128(r, c & 7)) =
        make_uint4(out[0], out[1], out[2], out[3]);
  }
}

template <int D>
__device__ __forceinline__ void zero_row(uint8_t* tile, int r) {
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {
    *reinterpret_cast<uint4*>(tile + (c >> 3) * kHalf + sw128(r, c & 7)) = make_uint4(0, 0, 0, 0);
  }
}

// 16 extension columns of one row.  A rank-G term sum_g a_jg * b_ig enters the
// score as three columns per group: (hi, hi, lo) of a on the query side
// against (hi, lo, hi) of b on the key side (FP16 high/low splits), so the
// column products sum to a * b to ~2^-21 relative.  Extension tile 0 holds
// the Jensen bias (a = -(scale/24) ||q'_g||^2, b = D_g^2), tile 1 the
// zero-point term of the keys (a = sum of q'_g, b = -z_g * D_g).
__device__ __forceinline__ void write_ext_row(uint8_t* tile, int r, const float* cols16) {
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = pack_h2(cols16[2 * i], cols16[2 * i + 1]);
  *reinterpret_cast<uint4*>(tile + noswz16(r, 0)) = make_uint4(w[0], w[1], w[2], w[3]);
  *reinterpret_cast<uint4*>(tile + noswz16(r, 1)) = make_uint4(w[4], w[5], w[6], w[7]);
}

__device__ __forceinline__ void split_h(float v, float& hi, float& lo) {
  hi = __half2float(__float2half_rn(v));
  lo = __half2float(__float2half_rn(v - hi));
}

template <int D, int BITS, int GROUP>
__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qlo,
                const __grid_constant__ CUtensorMap tm_qo, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using L = Smem<D>;
  constexpr int G = D / GROUP;
  constexpr int NKH = D / 64;            // 64-channel halves of a row
  constexpr int CB = D * BITS / 8;       // packed bytes per token
  constexpr int NW = CB / 4;             // packed words per token
  static_assert(3 * G <= 16, "bias columns");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int q0 = blockIdx.x * kBlockM;
  const int bh = blockIdx.y;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  const uint32_t bar_load = ptx::smem_u32(&bars[0]);
  const uint32_t bar_mma = ptx::smem_u32(&bars[1]);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBar + 16);

  const uint32_t s_q = ptx::smem_u32(smem + L::kQ);
  const uint32_t s_qlo = ptx::smem_u32(smem + L::kQlo);
  const uint32_t s_qo = ptx::smem_u32(smem + L::kQo);
  const bool precise = p.precise_query != 0;
  const uint32_t s_k = ptx::smem_u32(smem + L::kK);
  const uint32_t s_v = ptx::smem_u32(smem + L::kV);
  const uint32_t s_p = ptx::smem_u32(smem + L::kP);
  const uint32_t s_qx = ptx::smem_u32(smem + L::kQx);
  const uint32_t s_kx = ptx::smem_u32(smem + L::kKx);

  if (tid == 0) {
    ptx::mbar_init(bar_load, 1);
    ptx::mbar_init(bar_mma, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 256);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t t_s = tmem;              // S: columns [0, 128)
  const uint32_t t_o = tmem + 128;        // O: columns [128, 128 + D)

  uint32_t ph_load = 0, ph_mma = 0;
  const unsigned long long lim = p.wait_limit_ns;

  // ---- query tiles by TMA: rotated FP16 (+ low part), original BF16 ----
  if (tid == 0) {
    const int n_tiles = 1 + (precise ? 1 : 0) + (p.n_r > 0 ? 1 : 0);
    ptx::mbar_expect_tx(bar_load, n_tiles * NKH * kHalf);
#pragma unroll
    for (int h = 0; h < NKH; ++h) {
      ptx::tma_load_3d(s_q + h * kHalf, &tm_q, 64 * h, q0, bh, bar_load);
      if (precise) ptx::tma_load_3d(s_qlo + h * kHalf, &tm_qlo, 64 * h, q0, bh, bar_load);
      if (p.n_r > 0) ptx::tma_load_3d(s_qo + h * kHalf, &tm_qo, 64 * h, q0, bh, bar_load);
    }
  }
  bool ok = wait_bounded(bar_load, ph_load, lim);
  ph_load ^= 1;

  // ---- per-row group norms n_g = ||q'_g||^2, group sums, extension columns ----
  {
    float nrm[G], qsum[G];
#pragma unroll
    for (int g = 0; g < G; ++g) nrm[g] = qsum[g] = 0.f;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      const int off = (c >> 3) * kHalf + sw128(tid, c & 7);
      const uint4 v = *reinterpret_cast<const uint4*>(smem + L::kQ + off);
      uint4 vl = make_uint4(0u, 0u, 0u, 0u);
      if (precise) vl = *reinterpret_cast<const uint4*>(smem + L::kQlo + off);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      const uint32_t wl[4] = {vl.x, vl.y, vl.z, vl.w};
      float acc = 0.f, sum = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = h_lo(w[i]) + h_lo(wl[i]), b = h_hi(w[i]) + h_hi(wl[i]);
        acc = fmaf(a, a, acc);
        acc = fmaf(b, b, acc);
        sum += a + b;
      }
      nrm[(8 * c) / GROUP] += acc;
      qsum[(8 * c) / GROUP] += sum;
    }
    float cols[16], cols_z[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) cols[i] = cols_z[i] = 0.f;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float hi, lo;
      split_h(p.alpha_coef * nrm[g], hi, lo);
      cols[3 * g] = hi;
      cols[3 * g + 1] = hi;
      cols[3 * g + 2] = lo;
      split_h(qsum[g], hi, lo);
      cols_z[3 * g] = hi;
      cols_z[3 * g + 1] = hi;
      cols_z[3 * g + 2] = lo;
    }
    write_ext_row(smem + L::kQx, tid, cols);
    write_ext_row(smem + L::kQx + 4096, tid, cols_z);
    ptx::fence_proxy_async_smem();
  }

  const int n_ct = (p.n_s + kBlockN - 1) / kBlockN;
  const int n_rt = (p.n_r + kBlockN - 1) / kBlockN;
  const bool use_bias = p.corr != 0;
  const bool do_pv = !p.mass_only;
  constexpr uint32_t kIdescS = ptx::idesc_f16kind(kBlockM, kBlockN, false, false);
  constexpr uint32_t kIdescSbf = ptx::idesc_f16kind(kBlockM, kBlockN, false, true);
  constexpr uint32_t kIdescO = ptx::idesc_f16kind(kBlockM, D, true, false);

  float m_run = -INFINITY, l_s = 0.f, l_r = 0.f;
  const size_t head_tok = static_cast<size_t>(bh) * p.cap;

  for (int it = 0; it < n_ct + n_rt; ++it) {
    if (!__syncthreads_and(ok)) {
      ok = false;
      break;
    }
    const bool cached = it < n_ct;
    const int key0 = cached ? it * kBlockN : (it - n_ct) * kBlockN;
    const int n_valid = min(kBlockN, (cached ? p.n_s : p.n_r) - key0);

    if (cached) {
      // ---- dequantize key row `tid` of this tile into sK / sV / sKx ----
      const bool valid = tid < n_valid;
      if (valid) {
        const size_t tok = head_tok + key0 + tid;
        uint32_t kw[NW], ksz[G > 0 ? G : 1];
        const uint4* kc = reinterpret_cast<const uint4*>(p.k_codes + tok * CB);
#pragma unroll
        for (int i = 0; i < NW / 4; ++i) {
          const uint4 v = __ldg(kc + i);
          kw[4 * i] = v.x; kw[4 * i + 1] = v.y; kw[4 * i + 2] = v.z; kw[4 * i + 3] = v.w;
        }
#pragma unroll
        for (int g = 0; g < G; ++g) ksz[g] = __ldg(p.k_sz + tok * G + g);
        dequant_row<D, BITS, GROUP, false>(kw, ksz, smem + L::kK, tid);
        float cols[16], cols_z[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) cols[i] = cols_z[i] = 0.f;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float dl = bf16_lo(ksz[g]);
          float hi, lo;
          split_h(dl * dl, hi, lo);
          cols[3 * g] = hi;
          cols[3 * g + 1] = lo;
          cols[3 * g + 2] = hi;
          split_h(-bf16_hi(ksz[g]) * dl, hi, lo);
          cols_z[3 * g] = hi;
          cols_z[3 * g + 1] = lo;
          cols_z[3 * g + 2] = hi;
        }
        write_ext_row(smem + L::kKx, tid, cols);
        write_ext_row(smem + L::kKx + 4096, tid, cols_z);
        if (do_pv) {
          uint32_t vw[NW], vsz[G > 0 ? G : 1];
          const uint4* vc = reinterpret_cast<const uint4*>(p.v_codes + tok * CB);
#pragma unroll
          for (int i = 0; i < NW / 4; ++i) {
            const uint4 v = __ldg(vc + i);
            vw[4 * i] = v.x; vw[4 * i + 1] = v.y; vw[4 * i + 2] = v.z; vw[4 * i + 3] = v.w;
          }
#pragma unroll
          for (int g = 0; g < G; ++g) vsz[g] = __ldg(p.v_sz + tok * G + g);
          dequant_row<D, BITS, GROUP, true>(vw, vsz, smem + L::kV, tid);
        }
      } else {
        zero_row<D>(smem + L::kK, tid);
        if (do_pv) zero_row<D>(smem + L::kV, tid);
        const float zeros[16] = {0.f};
        write_ext_row(smem + L::kKx, tid, zeros);
        write_ext_row(smem + L::kKx + 4096, tid, zeros);
      }
      ptx::fence_proxy_async_smem();
      __syncthreads();
    } else {
      if (tid == 0) {
        ptx::mbar_expect_tx(bar_load, (do_pv ? 2 : 1) * NKH * kHalf);
#pragma unroll
        for (int h = 0; h < NKH; ++h) {
          ptx::tma_load_3d(s_k + h * kHalf, &tm_k, 64 * h, key0, bh, bar_load);
          if (do_pv) ptx::tma_load_3d(s_v + h * kHalf, &tm_v, 64 * h, key0, bh, bar_load);
        }
      }
      ok = wait_bounded(bar_load, ph_load, lim);
      ph_load ^= 1;
      if (!__syncthreads_and(ok)) {
        ok = false;
        break;
      }
    }

    // ---- S = Q' K_hat'^T (+ low part, + bias columns) or Q K^T ----
    if (tid == 0) {
      ptx::tc_fence_after();
      const uint32_t a_base = cached ? s_q : s_qo;
      const uint32_t idesc = cached ? kIdescS : kIdescSbf;
#pragma unroll
      for (int s = 0; s < D / 16; ++s) {
        const uint32_t off = (s >> 2) * kHalf + (s & 3) * 32;
        ptx::mma_f16(t_s, ptx::smem_desc(a_base + off, 16, 1024, ptx::kLayoutSw128),
                      ptx::smem_desc(s_k + off, 16, 1024, ptx::kLayoutSw128), idesc, s > 0);
      }
      if (cached && precise) {
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
          const uint32_t off = (s >> 2) * kHalf + (s & 3) * 32;
          ptx::mma_f16(t_s, ptx::smem_desc(s_qlo + off, 16, 1024, ptx::kLayoutSw128),
                        ptx::smem_desc(s_k + off, 16, 1024, ptx::kLayoutSw128), kIdescS, 1);
        }
      }
      if (cached) {
        // zero-point term of the keys, then (with the correction) the bias
        ptx::mma_f16(t_s, ptx::smem_desc(s_qx + 4096, 128, 256, ptx::kLayoutNone),
                      ptx::smem_desc(s_kx + 4096, 128, 256, ptx::kLayoutNone), kIdescS, 1);
        if (use_bias)
          ptx::mma_f16(t_s, ptx::smem_desc(s_qx, 128, 256, ptx::kLayoutNone),
                        ptx::smem_desc(s_kx, 128, 256, ptx::kLayoutNone), kIdescS, 1);
      }
      ptx::mma_commit(bar_mma);
    }
    ok = wait_bounded(bar_mma, ph_mma, lim);
    ph_mma ^= 1;
    ptx::tc_fence_after();

    // ---- online softmax of row tid ----
    float sc[kBlockN];
#pragma unroll
    for (int c = 0; c < kBlockN / 32; ++c) {
      uint32_t r[32];
      ptx::tmem_ld32(t_s + lane_off + 32 * c, r);
#pragma unroll
      for (int j = 0; j < 32; ++j) sc[32 * c + j] = __uint_as_float(r[j]);
    }
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < kBlockN; ++j) mx = (j < n_valid) ? fmaxf(mx, sc[j]) : mx;
    const float m_new = fmaxf(m_run, mx * p.scale_log2);
    const float alpha = exp2f(m_run - m_new);
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < kBlockN; ++j) {
      const float e = (j < n_valid) ? exp2f(fmaf(sc[j], p.scale_log2, -m_new)) : 0.f;
      sc[j] = e;
      sum += e;
    }
    l_s *= alpha;
    l_r *= alpha;
    if (cached) l_s += sum; else l_r += sum;
    m_run = m_new;

    if (do_pv) {
      // P (FP16) into the swizzled A tile, row tid
#pragma unroll
      for (int c = 0; c < kBlockN / 8; ++c) {
        const uint4 v = make_uint4(pack_h2(sc[8 * c], sc[8 * c + 1]),
                                   pack_h2(sc[8 * c + 2], sc[8 * c + 3]),
                                   pack_h2(sc[8 * c + 4], sc[8 * c + 5]),
                                   pack_h2(sc[8 * c + 6], sc[8 * c + 7]));
        *reinterpret_cast<uint4*>(smem + L::kP + (c >> 3) * kHalf + sw128(tid, c & 7)) = v;
      }
      // rescale the running output when the max moved (warp-uniform decision)
      if (it > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          ptx::tmem_ld32(t_o + lane_off + 32 * c, r);
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
          ptx::tmem_st32(t_o + lane_off + 32 * c, r);
        }
        ptx::tmem_st_wait();
      }
      ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before();
    __syncthreads();

    if (do_pv) {
      // ---- O += P V ----
      if (tid == 0) {
        ptx::tc_fence_after();
#pragma unroll
        for (int s = 0; s < kBlockN / 16; ++s) {
          const uint32_t a_off = (s >> 2) * kHalf + (s & 3) * 32;
          const uint32_t b_off = s * 16 * 128;
          ptx::mma_f16(t_o, ptx::smem_desc(s_p + a_off, 16, 1024, ptx::kLayoutSw128),
                        ptx::smem_desc(s_v + b_off, kHalf, 1024, ptx::kLayoutSw128), kIdescO,
                        (it > 0 || s > 0) ? 1u : 0u);
        }
        ptx::mma_commit(bar_mma);
      }
      ok = wait_bounded(bar_mma, ph_mma, lim) && ok;
      ph_mma ^= 1;
      ptx::tc_fence_after();
    }
  }

  // ---- epilogue ----
  ok = __syncthreads_and(ok) != 0;
  if (ok) {
    const float denom = l_s + l_r;
    const float inv = 1.0f / denom;
    const int row = q0 + tid;
    const bool row_ok = row < p.n_q;
    if (do_pv) {
      float o[D];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        ptx::tmem_ld32(t_o + lane_off + 32 * c, r);
#pragma unroll
        for (int j = 0; j < 32; ++j) o[32 * c + j] = __uint_as_float(r[j]) * inv;
      }
      // O = H^T O' = (1/sqrt(d)) diag(sigma) Sylvester(d) O'
#pragma unroll
      for (int h = 1; h < D; h <<= 1) {
#pragma unroll
        for (int i = 0; i < D; ++i) {
          if ((i & h) == 0) {
            const float a = o[i], b = o[i + h];
            o[i] = a + b;
            o[i + h] = a - b;
          }
        }
      }
      if (row_ok) {
        uint16_t* dst = p.out + (static_cast<size_t>(bh) * p.n_q + row) * D;
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          float v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int ch = 8 * c + e;
            const float s = ((p.sign_bits[ch >> 5] >> (ch & 31)) & 1u) ? -p.inv_sqrt_d : p.inv_sqrt_d;
            v[e] = o[ch] * s;
          }
          *reinterpret_cast<uint4*>(dst + 8 * c) =
              make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                         pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
        }
      }
    }
    if (row_ok && p.p_s != nullptr) {
      p.p_s[static_cast<size_t>(bh) * p.n_q + row] = l_s * inv;
      p.p_r[static_cast<size_t>(bh) * p.n_q + row] = l_r * inv;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 256);
  }
}

__global__ void wait_selftest_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = ptx::smem_u32(&bar);
  if (threadIdx.x == 0) {
    ptx::mbar_init(b, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  // nothing ever arrives on this barrier: the wait must run out and return
  wait_bounded(b, 0, limit_ns);
}

// ---- host side -------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
  });
  return fn;
}

// 3-D map over a [bh][n][d] 16-bit tensor, box [1][128][64], 128-byte
// swizzle, zero fill outside the tensor.
bool make_map(CUtensorMap* m, const void* base, int d, int n, int bh, bool bf16) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)n, (cuuint64_t)bh};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)n * d * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, int BITS, int GROUP>
kvq_status launch_t(const AttnLaunch& a, cudaStream_t stream) {
  using L = Smem<D>;
  static bool attr_set = false;
  auto kern = attn_kernel<D, BITS, GROUP>;
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc) !=
        cudaSuccess)
      return KVQ_ERR_CUDA;
    attr_set = true;
  }
  CUtensorMap mq, mqlo, mqo, mk, mv;
  if (!make_map(&mq, a.q_rot, D, a.n_q, a.bh, false)) return KVQ_ERR_CUDA;
  if (!make_map(&mqlo, a.q_rot_lo, D, a.n_q, a.bh, false)) return KVQ_ERR_CUDA;
  if (!make_map(&mqo, a.q_orig, D, a.n_q, a.bh, true)) return KVQ_ERR_CUDA;
  if (a.n_r > 0) {
    if (!make_map(&mk, a.k_cur, D, a.n_r, a.bh, true)) return KVQ_ERR_CUDA;
    if (a.mass_only) {
      mv = mk;
    } else if (!make_map(&mv, a.v_rot, D, a.n_r, a.bh, false)) {
      return KVQ_ERR_CUDA;
    }
  } else {
    mk = mq;
    mv = mq;
  }
  AttnParams p;
  p.k_codes = a.k_codes;
  p.v_codes = a.v_codes;
  p.k_sz = a.k_sz;
  p.v_sz = a.v_sz;
  p.n_s = a.n_s;
  p.cap = a.cap;
  p.n_q = a.n_q;
  p.n_r = a.n_r;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.alpha_coef = a.corr ? -(a.scale / 24.0f) : 0.0f;
  p.corr = a.corr;
  p.precise_query = a.precise_query;
  p.mass_only = a.mass_only;
  p.out = a.out;
  p.p_s = a.p_s;
  p.p_r = a.p_r;
  for (int i = 0; i < 4; ++i) p.sign_bits[i] = a.sign_bits[i];
  p.inv_sqrt_d = (float)(1.0 / sqrt((double)D));
  p.wait_limit_ns = a.wait_limit_ns;
  dim3 grid((a.n_q + kBlockM - 1) / kBlockM, a.bh);
  kern<<<grid, kThreads, L::kAlloc, stream>>>(mq, mqlo, mqo, mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace

kvq_status launch_attention(const AttnLaunch& a, int d, int bits, int group, cudaStream_t stream) {
#define KVQ_A(D_, B_, G_) \
  if (d == D_ && bits == B_ && group == G_) return launch_t<D_, B_, G_>(a, stream);
  KVQ_A(64, 2, 32)
  KVQ_A(64, 4, 32)
  KVQ_A(64, 2, 64)
  KVQ_A(64, 4, 64)
  KVQ_A(128, 2, 32)
  KVQ_A(128, 4, 32)
  KVQ_A(128, 2, 64)
  KVQ_A(128, 4, 64)
#undef KVQ_A
  return KVQ_ERR_UNSUPPORTED;
}

kvq_status read_and_clear_attention_status(int* status) {
  int zero = 0;
  if (cudaMemcpyFromSymbol(status, g_attn_status, sizeof(int)) != cudaSuccess) return KVQ_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(int)) != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cudaGetLastError();
}

}  // namespace kvq
