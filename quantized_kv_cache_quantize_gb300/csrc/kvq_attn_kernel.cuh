// Fused Jensen-bias-corrected chunk attention over a low-bit KV window
// (sm_103a: TMA, tcgen05 MMA with tensor-memory accumulators, warp
// specialization).
//
// Paper: "Quantized Keys Steal Attention" -- abstract and section 1 (the
// current chunk attends over the cached window and itself; a per-score
// correction b, from the cached keys' step sizes and the query norm, is
// subtracted before the softmax from cached-key scores only), Figure 3
// caption (b removes the Jensen bias E[exp(s + delta)] > exp(s)), section 3
// (Eq. (1) dequantization, Hadamard rotation), Figure 2 caption (the masses
// P_S and P_R).
//
// One CTA owns NQ tiles of 128 query rows of one (batch, head) and walks the
// key tiles (128 keys) of the cached window, then of the current chunk.
// Roles (warps):
//   softmax   NQ warpgroups; thread r of group q owns row r of query tile q
//             (TMEM lane r): online softmax with one running max and two
//             running sums (cached, current), P written back into TMEM;
//   dequant   one warpgroup; thread r turns key r of a cached tile into FP16
//             K and V rows in shared memory (128-byte swizzle) plus its
//             extension columns;
//   MMA       one thread issues every tcgen05.mma: S = Q K^T (both operands in
//             shared memory), O += P V (P from tensor memory);
//   TMA       one thread loads the query tiles and the current-chunk tiles.
// Hand-offs are mbarriers (two K/V stages, S ready, P ready, stage free);
// every wait is bounded by a time limit.
//
// Numerics.  Cached scores: the K tile holds code * D (INT2, <= 10
// significant bits) or (code - 8) * D (INT4, <= 11), exact in FP16; two rank-G
// terms enter through one 16-column extension tile contracted on the tensor
// core: the keys' zero points (sum_g (sum_{c in g} q'_c) * (o - z_g) D_g,
// o the code offset, three columns per group, FP16
// high/low splits, so the products carry ~2^-21 relative error) and, with the
// correction, the Jensen bias -(scale/24) sum_g ||q'_g||^2 D_g^2 (one column
// per group, ~2^-11 relative error on a term that is a small fraction of the
// score; with the precise-query flag a second extension tile carries it with
// three columns per group as well).  The rotated
// query is FP16 (or FP16 high + low parts with the precise-query flag: one
// more QK pass on cached tiles).  Current scores use the BF16 inputs as they
// are (exact products).  P and the rotated current values are FP16; V tiles
// hold (code - z) * D rounded once to FP16.  Limits: |values| < 65504 after
// rotation, step sizes < 4096.
//
// Kernel templates and their host-side launch, shared by the translation
// units that instantiate them (kvq_attn.cu, kvq_attn_exact.cu,
// kvq_attn_kch.cu), so that the instances compile in parallel.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "kvq_checks.cuh"
#include "kvq_fwht.cuh"
#include "kvq_tmap.cuh"
#include "kvq_internal.h"
#include "kvq_sm100.cuh"

namespace kvq {

namespace {

struct AttnParams {
  const uint8_t* k_codes;
  const uint8_t* v_codes;
  const uint32_t* k_sz;
  const uint32_t* v_sz;
  int n_s, cap, n_q, n_r;
  float scale_log2;   // scale * log2(e)
  float alpha_coef;   // -(scale / 24) * 2^8 with the Taylor correction, 0 otherwise
  float half_scale;   // scale / 2 (exact correction: a_c = half_scale * |q'_c| * D)
  int corr;
  int mass_only;
  uint16_t* out;
  float* p_s;
  float* p_r;
  uint32_t sign_bits[4];
  float inv_sqrt_d;
  unsigned long long wait_limit_ns;
  // key-range split (blockIdx.z = split): each CTA walks key tiles
  // [z * tiles_per_split, ...) of the cached tiles followed by the current
  // ones; with o_part set it leaves partial results for the merge kernel
  int tiles_per_split;
  float* o_part;    // [splits][B*H][n_q][D] fp32, unnormalized, rotated basis
  float* st_part;   // [splits][B*H][n_q][3]: base m (log2 units), l_S, l_R
  // per-channel keys: cached tile t is block t % bpc of chunk slot t / bpc;
  // k_sz holds kblk_per_head blocks of D (step, zero) words per head;
  // kch_c [B*H][n_ct][n_q]: zero-point term minus correction per query row
  // and tile (log2 units)
  int chunk, bpc, kblk_per_head, n_ct;
  const float* kch_c;
  int* status;      // device status word (first error of a bounded wait)
  int* bounds_site; // checked build: source line of the first failed index check
  // per-head kernel choice (two kernels share one call): select = 0 runs
  // every (batch, head); +1 only the heads whose precise-query criterion
  // holds, -1 only the others (criterion: select_scale * sqrt(qn2 * kn2)
  // >= kPreciseSelect)
  int select;
  float select_scale;
  const float* qn2;
  const float* kn2;
};

// whether this CTA's (batch, head) belongs to the other kernel of the call
__device__ __forceinline__ bool head_not_mine(const AttnParams& p, int bh) {
  if (p.select == 0) return false;
  const bool precise = !(p.select_scale * sqrtf(p.qn2[bh] * p.kn2[bh]) < kPreciseSelect);
  return precise != (p.select > 0);
}

constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
constexpr int kHalf = 16384;   // one [128 rows][64 x 16-bit] swizzled sub-tile
constexpr int kExt = 4096;     // one [128 rows][16 x 16-bit] tile, no swizzle
constexpr float kChunkSumLimit = 32768.0f;  // 2^15: every P of the chunk stays FP16
constexpr float kF16Max = 65504.0f;

// Extension-column scalings keeping every FP16 operand in range: bias
// a * 2^8 against D^2 * 2^-8, zero-point term q-sum * 2^4 against -z D * 2^-4.
constexpr float kBiasKeyScale = 1.0f / 256.0f;
constexpr float kZeroQueryScale = 16.0f;
constexpr float kZeroKeyScale = 1.0f / 16.0f;

// With KVQ_FLAG_STAGED_WORDS the default form (head_dim 128, INT2 groups of
// 32, two query tiles per CTA, no precise split, exact term or per-channel
// keys) stages the packed codes and (step, zero) words of the cached tiles
// into shared memory with bulk copies (TMA), one tile ahead; the other forms
// have no shared memory left for it.  Without the flag (the default, 7 %
// faster as measured) every form loads them per thread, a tile ahead, into
// registers.
template <int D, int BITS, int GROUP, int NQ, bool PRECISE, bool EXACT, bool KCH>
__host__ __device__ constexpr bool codes_by_tma() {
  return D == 128 && BITS == 2 && GROUP == 32 && NQ == 2 && !PRECISE && !EXACT && !KCH;
}

template <int D, int NQ, bool PRECISE, bool EXACT, bool KCH, bool CODES_TMA = false>
struct Cfg {
  static constexpr int kTile = kBlockM * D * 2;
  static constexpr int kNKH = D / 64;
  static constexpr int kSBuf = NQ == 1 ? 2 : 1;            // S buffers per query tile
  // shared memory
  static constexpr int kQ = 0;                             // NQ hi tiles [, NQ lo tiles]
  static constexpr int kQx = kQ + NQ * kTile * (PRECISE ? 2 : 1);
  static constexpr int kNExt = PRECISE ? 2 : 1;              // extension tiles
  // exact correction: per stage [4 groups][128 keys] fp32 (scale * D / 2)^2,
  // then [4 groups][4 warps] maxima over the tile; padded so that both
  // stages stay 1024-byte aligned
  static constexpr int kDsq = 2 * kTile + kNExt * kExt;    // offset inside a stage
  static constexpr int kDsqBytes = EXACT ? 3072 : 0;
  // per-channel keys: per stage the key block's steps (FP16, [128]) and
  // -magic * steps (FP16, [128]), padded like dsq
  static constexpr int kKch = kDsq + kDsqBytes;
  static constexpr int kKchBytes = KCH ? 1024 : 0;
  static constexpr int kStageBytes = 2 * kTile + kNExt * kExt + kDsqBytes + kKchBytes;  // K, V, Kx [, dsq] [, kch]
  static constexpr int kStages = kQx + NQ * kNExt * kExt;
  // staged key and value words of one cached tile (CODES_TMA): per half the
  // codes [128 keys][32 B], then the (step, zero) words [128 keys][16 B]
  static constexpr int kCodes = kStages + 2 * kStageBytes;
  static constexpr int kCodeHalf = 128 * 32 + 128 * 16;
  static constexpr int kCodeBytes = CODES_TMA ? 2 * kCodeHalf : 0;
  static constexpr int kBar = kCodes + kCodeBytes;
  static constexpr int kBytes = kBar + 256;
  static constexpr int kAlloc = kBytes + 1024;
  // warps
  static constexpr int kSoftmaxWarps = 4 * NQ;
  static constexpr int kDequantWarp = kSoftmaxWarps;
  static constexpr int kMmaWarp = kSoftmaxWarps + 4;
  static constexpr int kThreads = (kSoftmaxWarps + 6) * 32;
  // tensor memory columns: S buffers, then the O tiles
  static constexpr int kTO = NQ * kSBuf * 128;
  static constexpr int kTQ = kTO + NQ * D;   // exact correction: the row's rotated query, fp32
  static constexpr int kTCols = 512;
  static_assert(kTO + NQ * D * (EXACT ? 2 : 1) <= kTCols, "tensor memory");
  static_assert(!EXACT || NQ == 1, "exact correction: one query tile per CTA");
  static_assert(!(EXACT && KCH), "per-channel keys take the exact correction from the pre-pass");
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
  static_assert(kAlloc <= 232448, "shared memory");
};

// mbarrier slots
//
// A cached stage is handed over in two parts: its K half (key rows and
// extension rows) and its V half (value rows, and the exact correction's
// per-key step terms).  The K half is free again once both query tiles'
// QK MMAs of the tile are done, the V half once their PV MMAs are, so the
// dequant warps can fill the next K half about a tile period before the MMA
// needs it instead of in the gap between the last PV and the next QK.
enum : int {
  kBarQ = 0,        // query tiles landed (phase 0: rotated, phase 1: original)
  kBarQFree = 1,    // all cached-tile QK MMAs done: query buffers reusable
  kBarQx = 2,       // query extension columns written (NQ * 128 arrivals)
  kBarFullK = 3,    // [2] cached stage: K half dequantized (128 arrivals)
  kBarFullTma = 5,  // [2] current stage loaded (TMA)
  kBarEmptyV = 7,   // [2] stage's V half consumed (MMA commit after the last PV)
  kBarS = 9,        // [2] S buffer ready (MMA commit)
  kBarP = 11,       // [NQ] P written, O rescaled (128 arrivals)
  kBarOStep = 13,   // [NQ] PV of a tile done (MMA commit; one-tile schedule)
  kBarODone = 15,   // [NQ] every MMA done (MMA commit)
  kBarKch = 17,     // [2] per-channel keys: the stage's block steps written (128 arrivals)
  kBarFullV = 19,   // [2] cached stage: V half dequantized (128 arrivals)
  kBarEmptyK = 21,  // [2] stage's K half consumed (MMA commit after the last QK)
  kBarCodeK = 23,   // staged key words of the next cached tile landed (bulk copies)
  kBarCodeKFree = 24,  // those words read by the dequant warps (128 arrivals)
  kBarCodeV = 25,   // staged value words landed
  kBarCodeVFree = 26,  // value words read (128 arrivals)
  kBarCount = 27
};
constexpr int kAbortOffset = kBarCount * 8;
constexpr int kTmemSlotOffset = kAbortOffset + 4;

// Bounded wait on an mbarrier phase: false when the time limit ran out (the
// status word and the CTA's abort flag are set) or another role aborted.
__device__ bool wait_bar(uint32_t bar, uint32_t parity, unsigned long long limit_ns,
                         volatile int* abort, int* status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  // suspended in the wait instruction (up to 20 us per try) instead of
  // spinning: waiting warps leave the issue slots to the working ones
  while (!ptx::mbar_try_wait_sleep(bar, parity, 20000u)) {
    if (*abort) return false;
    if (ptx::globaltimer() - t0 > limit_ns) {
      *abort = 1;
      atomicCAS(status, 0, (int)KVQ_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// byte offset of 16-byte chunk `c` (0..7) of row `r` in a 128-byte-swizzled
// [rows][64 x 16-bit] sub-tile
__device__ __forceinline__ int sw128(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

// byte offset of 16-byte K-chunk `kc` (0..1) of row r of a [128][16] 16-bit
// K-major tile without swizzle: 8-row x 16-byte core matrices, K chunks
// 128 B apart, row groups 256 B apart
__device__ __forceinline__ int noswz16(int r, int kc) {
  return (r >> 3) * 256 + kc * 128 + (r & 7) * 16;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float h_lo(uint32_t w) {
  return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu)));
}
__device__ __forceinline__ float h_hi(uint32_t w) {
  return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ __half2 as_h2(uint32_t w) { return *reinterpret_cast<__half2*>(&w); }
__device__ __forceinline__ uint32_t as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

__device__ __forceinline__ void split_h(float v, float& hi, float& lo) {
  hi = __half2float(__float2half_rn(v));
  lo = __half2float(__float2half_rn(v - hi));
}

// 16 extension columns of one row.  Merged tile: columns [0, G) hold the
// bias factors of the G groups (query side a_g, key side b_g), columns
// G + 3g .. G + 3g + 2 the zero-point factors of group g as (hi, hi, lo) on the
// query side against (hi, lo, hi) on the key side.  Precise layout: tile 0 the
// bias factors split the same way in columns 3g .. 3g + 2, tile 1 the
// zero-point factors in columns 3g .. 3g + 2.  Unused columns are zero.
__device__ __forceinline__ void write_ext_row(uint8_t* tile, int r, const float (&cols)[16]) {
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = pack_h2(cols[2 * i], cols[2 * i + 1]);
  *reinterpret_cast<uint4*>(tile + noswz16(r, 0)) = make_uint4(w[0], w[1], w[2], w[3]);
  *reinterpret_cast<uint4*>(tile + noswz16(r, 1)) = make_uint4(w[4], w[5], w[6], w[7]);
}

// The code pair k of a packed word (low code at bit BITS*k, high code 16 bits
// up), ORed into an FP16 constant of each half so that the half reads
// exactly magic + code.  INT2: a code at bits [6, 8) of a half under 16.0
// (0x4C00, unit 1/64) or at bits [8, 10) under 4.0 (0x4400, unit 1/256) has
// weight 1, so one shifted copy of the word serves two pairs: w << 6 (pairs
// 0, 1), w << 2 (2), w (3, 4), w >> 4 (5, 6), w >> 8 (7); four shifts per
// word.  INT4: bits [6, 10) under 16.0, one shift per pair.
template <int BITS>
__device__ __forceinline__ int pair_magic(int k) {   // 16 or 4
  return BITS == 4 ? 16 : ((k == 1 || k == 4 || k == 6) ? 4 : 16);
}
template <int BITS>
__device__ __forceinline__ uint32_t code_pair_f16(uint32_t w, int k) {
  if (BITS == 4) {
    const int pos = 4 * k;
    const uint32_t t = pos <= 6 ? (w << (6 - pos)) : (w >> (pos - 6));
    return (t & 0x03C003C0u) | 0x4C004C00u;
  }
  const uint32_t t = k <= 1 ? (w << 6) : k == 2 ? (w << 2) : k <= 4 ? w : k <= 6 ? (w >> 4) : (w >> 8);
  return pair_magic<2>(k) == 4 ? ((t & 0x03000300u) | 0x44004400u) : ((t & 0x00C000C0u) | 0x4C004C00u);
}

// Code offset of the key tiles: an INT4 key tile holds (code - 8) * D, whose
// magnitude needs at most 3 significant bits times the 8 of the BF16 step (11
// bits: exact in FP16, where code * D can need 12); the zero-point term
// carries (8 - z) * D instead of -z * D.  INT2 codes need no offset.
template <int BITS>
__device__ __forceinline__ constexpr int key_code_offset() { return BITS == 4 ? 8 : 0; }

// Dequantize one packed key row into row r of a swizzled FP16 tile.
// ZERO = false (keys): (code - o) * D = (magic + code) D - (magic + o) D in
// one FMA, o the key code offset, exact.  ZERO = true (values): (code - z) * D, the integer
// difference exact, one rounding of the product.
template <int D, int BITS, int GROUP, bool ZERO>
__device__ __forceinline__ void dequant_row(const uint32_t (&words)[D * BITS / 32],
                                            const uint32_t (&sz)[D / GROUP], uint8_t* tile,
                                            int r) {
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {
    const int g = (8 * c) / GROUP;
    const __half2 d2 = __float2half2_rn(bf16_lo(sz[g]));
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int k = BITS == 2 ? 4 * (c & 1) + i : i;
      const float mg = (float)pair_magic<BITS>(k);
      const __half2 k2 = ZERO ? __float2half2_rn(mg + bf16_hi(sz[g]))
                              : __float2half2_rn(-(mg + (float)key_code_offset<BITS>()) * bf16_lo(sz[g]));
      const uint32_t v = BITS == 2 ? code_pair_f16<2>(words[c >> 1], k) : code_pair_f16<4>(words[c], k);
      const __half2 res = ZERO ? __hmul2(__hsub2(as_h2(v), k2), d2) : __hfma2(as_h2(v), d2, k2);
      out[i] = as_u32(res);
    }
    *reinterpret_cast<uint4*>(tile + (c >> 3) * kHalf + sw128(r, c & 7)) =
        make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// Per-channel keys: one packed key row into row r of a swizzled FP16 tile as
// (code - o) * D_c = (magic + code) D_c - (magic + o) D_c in one FMA, o the
// key code offset, exact (the zero-point term goes to the per-(row, tile)
// pre-pass): kd holds the block's steps D_c, kmd the constants
// -(magic + o) D_c (FP16, one per channel; magic as code_pair_f16 places the
// pair)
template <int D, int BITS>
__device__ __forceinline__ void dequant_row_kch(const uint32_t (&words)[D * BITS / 32],
                                                const uint8_t* kd, const uint8_t* kmd,
                                                uint8_t* tile, int r) {
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {
    const uint4 dv = *reinterpret_cast<const uint4*>(kd + 16 * c);
    const uint4 mv = *reinterpret_cast<const uint4*>(kmd + 16 * c);
    const uint32_t d2[4] = {dv.x, dv.y, dv.z, dv.w};
    const uint32_t m2[4] = {mv.x, mv.y, mv.z, mv.w};
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int k = BITS == 2 ? 4 * (c & 1) + i : i;
      const uint32_t v = BITS == 2 ? code_pair_f16<2>(words[c >> 1], k) : code_pair_f16<4>(words[c], k);
      out[i] = as_u32(__hfma2(as_h2(v), as_h2(d2[i]), as_h2(m2[i])));
    }
    *reinterpret_cast<uint4*>(tile + (c >> 3) * kHalf + sw128(r, c & 7)) =
        make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// Exponentials of one 32-column chunk of scores against the base m: P pairs
// in FP16 (low column in the low half) and the packed pair of partial sums;
// with MASKED, columns at or past `valid` give 0 (the last tile of a
// segment; every other tile takes the unmasked form, which has no per-column
// compare and select).
template <bool MASKED>
__device__ __forceinline__ uint64_t exp_chunk(const uint32_t (&s)[32], uint64_t sl2x2, float m,
                                              int valid, uint32_t (&pk)[16]) {
  const uint64_t negm2 = ptx::f2_pack(-m, -m);
  uint64_t acc = ptx::f2_pack(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    float x0, x1;
    ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[2 * k]), __uint_as_float(s[2 * k + 1])),
                               sl2x2, negm2),
                   x0, x1);
    float e0 = ptx::ex2_approx(x0);
    float e1 = ptx::ex2_approx(x1);
    if (MASKED && valid < 32) {
      e0 = (2 * k < valid) ? e0 : 0.f;
      e1 = (2 * k + 1 < valid) ? e1 : 0.f;
    }
    acc = ptx::f2_add(acc, ptx::f2_pack(e0, e1));
    pk[k] = ptx::f16x2_rn(e0, e1);
  }
  return acc;
}

// ---- exact correction -------------------------------------------------------
//
// For independent uniform noise on the cached key's rotated channels,
// E[exp(delta_ij)] = prod_c sinh(a_c) / a_c with a_c = (scale / 2) |q'_c| D_g(c),
// so the exact correction is b_ij = sum_c f(a_c), f(a) = log(sinh(a) / a).
// f has the power series f(a) = sum_k c_k a^(2k), c_k = 2^(2k) B_2k / (2k (2k)!)
// (B_2k the Bernoulli numbers), convergent for a < pi.  The kernels use a
// polynomial of the same form with kFitTerms terms p_k, the Chebyshev
// interpolant of f(a) / a^2 on a^2 in [0, kFitTmax] rewritten in powers of
// a^2 (sinhc_fit.py beside this header derives the constants): within
// 3e-7 of f per channel for a <= 3.  For one query row and group g with
// mu_g = max_{c in g} q'_c^2 and T = mu_g (scale D_g / 2)^2, the group's term
// is then sum_k p_k M_k T^k with the row's normalized moments
// M_k = sum_{c in g} (q'_c^2 / mu_g)^k: a polynomial in the key's T, valid
// while T <= kFitTmax (every a_c of the group <= 3).  Larger T takes the
// per-channel evaluation.
constexpr int kFitTerms = 8;
constexpr float kFitTmax = 9.0f;
__host__ __device__ constexpr float sinhc_fit(int k) {    // p_(k+1)
  return k == 0 ? 1.666666567e-01f
       : k == 1 ? -5.555371288e-03f
       : k == 2 ? 3.522899351e-04f
       : k == 3 ? -2.603568646e-05f
       : k == 4 ? 1.934644388e-06f
       : k == 5 ? -1.229594915e-07f
       : k == 6 ? 5.371698197e-09f
                : -1.124628862e-10f;
}
constexpr float kLog2e = 1.4426950408889634f;

// f(a) = log(sinh(a) / a) for a >= 0: the fitted polynomial for a <= 3
// (fused multiply-adds only), else a + log((1 - exp(-2a)) / (2a))
__device__ __forceinline__ float log_sinhc(float a) {
  const float t = a * a;
  if (t <= kFitTmax) {
    float p = sinhc_fit(kFitTerms - 1);
#pragma unroll
    for (int k = kFitTerms - 2; k >= 0; --k) p = fmaf(p, t, sinhc_fit(k));
    return p * t;
  }
  return a + __logf(__fdividef(1.0f - __expf(-2.0f * a), a + a));
}

// exp_chunk with a per-column additive term nb (log2 units, pairs packed):
// 2^(s * scale * log2(e) + nb - m)
template <bool MASKED>
__device__ __forceinline__ uint64_t exp_chunk_b(const uint32_t (&s)[32], const uint64_t (&nb)[16],
                                                uint64_t sl2x2, float m, int valid,
                                                uint32_t (&pk)[16]) {
  const uint64_t negm2 = ptx::f2_pack(-m, -m);
  uint64_t acc = ptx::f2_pack(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    float x0, x1;
    ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[2 * k]), __uint_as_float(s[2 * k + 1])),
                               sl2x2, ptx::f2_add(nb[k], negm2)),
                   x0, x1);
    float e0 = ptx::ex2_approx(x0);
    float e1 = ptx::ex2_approx(x1);
    if (MASKED && valid < 32) {
      e0 = (2 * k < valid) ? e0 : 0.f;
      e1 = (2 * k + 1 < valid) ? e1 : 0.f;
    }
    acc = ptx::f2_add(acc, ptx::f2_pack(e0, e1));
    pk[k] = ptx::f16x2_rn(e0, e1);
  }
  return acc;
}

// The exact correction of 32 cached keys for one query row, in log2 units
// and negated (nb = -log2(e) b), by the fitted polynomial: dq points at the
// chunk's (scale D_g / 2)^2 values ([group][128 keys] layout), mu2 / a2 hold
// the row's mu_g and -log2(e) p_k M_k as packed pairs.  Valid for the keys
// whose T = mu_g (scale D_g / 2)^2 <= kFitTmax in every group; the others get
// whatever the polynomial gives (exact_fix replaces them).
template <int G>
__device__ __forceinline__ void exact_series(const float* dq, const uint64_t (&mu2)[G],
                                             const uint64_t (&a2)[G][kFitTerms],
                                             uint64_t (&nb)[16]) {
#pragma unroll
  for (int k = 0; k < 16; ++k) nb[k] = 0ull;   // (+0, +0)
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int k4 = 0; k4 < 8; ++k4) {
      const float4 d4 = *reinterpret_cast<const float4*>(dq + g * kBlockN + 4 * k4);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint64_t t2 = ptx::f2_mul(mu2[g], h ? ptx::f2_pack(d4.z, d4.w) : ptx::f2_pack(d4.x, d4.y));
        uint64_t pp = a2[g][kFitTerms - 1];
#pragma unroll
        for (int i = kFitTerms - 2; i >= 0; --i) pp = ptx::f2_fma(pp, t2, a2[g][i]);
        nb[2 * k4 + h] = ptx::f2_fma(pp, t2, nb[2 * k4 + h]);
      }
    }
  }
}

// Keys of the chunk with T > kFitTmax in some group (some a_c above 3):
// their term is rebuilt from the polynomial of the other groups and, for the
// groups above the bound, the per-channel sum of log(sinh(a_c) / a_c) over
// the row's rotated query in tensor memory (t_q, fp32).  Warp-collective
// (tensor memory loads): called by whole warps.
template <int G, int D, int GROUP>
__device__ __noinline__ void exact_fix(const float* dq, const uint64_t (&mu2)[G],
                                       const uint64_t (&a2)[G][kFitTerms], uint32_t t_q,
                                       uint64_t (&nb)[16]) {
  float mu[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float unused;
    ptx::f2_unpack(mu2[g], mu[g], unused);
  }
  uint32_t vm[G];
  uint32_t any = 0;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    vm[g] = 0u;
#pragma unroll 4
    for (int k = 0; k < 32; ++k) vm[g] |= (mu[g] * dq[g * kBlockN + k] > kFitTmax ? 1u : 0u) << k;
    any |= vm[g];
  }
  if (!__any_sync(0xffffffffu, any != 0u)) return;
  float fix[32];
  // series part of the groups within the bound
#pragma unroll 1
  for (int k = 0; k < 32; ++k) {
    float acc = 0.f;
    if ((any >> k) & 1u) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float t = mu[g] * dq[g * kBlockN + k];
        if (t <= kFitTmax) {
          float a, unused;
          ptx::f2_unpack(a2[g][kFitTerms - 1], a, unused);
          float pp = a;
#pragma unroll
          for (int i = kFitTerms - 2; i >= 0; --i) {
            ptx::f2_unpack(a2[g][i], a, unused);
            pp = fmaf(pp, t, a);
          }
          acc = fmaf(pp, t, acc);
        }
      }
    }
    fix[k] = acc;
  }
  // per-channel terms of the groups above the bound, 32 channels at a time
  uint32_t vmr[G];
#pragma unroll
  for (int g = 0; g < G; ++g) vmr[g] = vm[g];
#pragma unroll 1
  for (int cb = 0; cb < D / 32; ++cb) {
    const int g = (32 * cb) / GROUP;
    uint32_t mk = 0u;
#pragma unroll
    for (int gg = 0; gg < G; ++gg) mk = gg == g ? vmr[gg] : mk;
    if (!__any_sync(0xffffffffu, mk != 0u)) continue;
    uint32_t qv[32];
    ptx::tmem_ld32(t_q + 32 * cb, qv);
    while (mk != 0u) {
      const int k = __ffs(mk) - 1;
      mk &= mk - 1u;
      const float dt = sqrtf(dq[g * kBlockN + k]);
      float sum = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) sum += log_sinhc(fabsf(__uint_as_float(qv[i])) * dt);
      fix[k] = fmaf(-kLog2e, sum, fix[k]);
    }
  }
#pragma unroll
  for (int k2 = 0; k2 < 16; ++k2) {
    float lo, hi;
    ptx::f2_unpack(nb[k2], lo, hi);
    if ((any >> (2 * k2)) & 1u) lo = fix[2 * k2];
    if ((any >> (2 * k2 + 1)) & 1u) hi = fix[2 * k2 + 1];
    nb[k2] = ptx::f2_pack(lo, hi);
  }
}

template <int D>
__device__ __forceinline__ void zero_row(uint8_t* tile, int r) {
#pragma unroll
  for (int c = 0; c < D / 8; ++c)
    *reinterpret_cast<uint4*>(tile + (c >> 3) * kHalf + sw128(r, c & 7)) = make_uint4(0, 0, 0, 0);
}

template <int D, int BITS, int GROUP, int NQ, bool PRECISE, bool EXACT, bool KCH, bool STAGED = false>
__global__ void __launch_bounds__(Cfg<D, NQ, PRECISE, EXACT, KCH>::kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qlo,
                const __grid_constant__ CUtensorMap tm_qo, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  constexpr bool kCodesTma = STAGED && codes_by_tma<D, BITS, GROUP, NQ, PRECISE, EXACT, KCH>();
  using C = Cfg<D, NQ, PRECISE, EXACT, KCH, kCodesTma>;
  constexpr int G = D / GROUP;
  constexpr int CB = D * BITS / 8;       // packed bytes per token
  constexpr int NW = CB / 4;             // packed words per token
  constexpr int NKH = C::kNKH;
  static_assert((PRECISE ? 3 : 4) * G <= 16, "extension columns");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int q0 = blockIdx.x * (kBlockM * NQ);
  const int bh = blockIdx.y;
  // a head the call gives to the other kernel: nothing set up yet, leave
  if (head_not_mine(p, bh)) return;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBar);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::kBar + kAbortOffset);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kBar + kTmemSlotOffset);
  const uint32_t bar0 = ptx::smem_u32(bars);
#define BAR(i) (bar0 + 8u * (uint32_t)(i))

  if (tid == 0) {
    ptx::mbar_init(BAR(kBarQ), 1);
    ptx::mbar_init(BAR(kBarQFree), 1);
    ptx::mbar_init(BAR(kBarQx), NQ * 128);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(BAR(kBarFullK + s), 128);
      ptx::mbar_init(BAR(kBarFullV + s), 128);
      ptx::mbar_init(BAR(kBarFullTma + s), 1);
      ptx::mbar_init(BAR(kBarEmptyK + s), 1);
      ptx::mbar_init(BAR(kBarEmptyV + s), 1);
      ptx::mbar_init(BAR(kBarS + s), 1);
      ptx::mbar_init(BAR(kBarP + s), 128);
      ptx::mbar_init(BAR(kBarOStep + s), 1);
      ptx::mbar_init(BAR(kBarODone + s), 1);
      ptx::mbar_init(BAR(kBarKch + s), 128);
    }
    ptx::mbar_init(BAR(kBarCodeK), 1);
    ptx::mbar_init(BAR(kBarCodeKFree), 128);
    ptx::mbar_init(BAR(kBarCodeV), 1);
    ptx::mbar_init(BAR(kBarCodeVFree), 128);
    *abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::kTCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // this CTA's key tiles: [jb, je) of the cached tiles followed by the
  // current ones; n_t, n_ct and every loop index below are local to the
  // range, kb and cb map them back to cached / current tile numbers
  const int n_ct_all = KCH ? p.n_ct : (p.n_s + kBlockN - 1) / kBlockN;
  const int n_t_all = n_ct_all + (p.n_r + kBlockN - 1) / kBlockN;
  const int jb = blockIdx.z * p.tiles_per_split;
  const int je = min(n_t_all, jb + p.tiles_per_split);
  const int n_t = max(0, je - jb);
  const int n_ct = max(0, min(n_ct_all, je) - jb);
  const int kb = jb;                        // cached tile = kb + j for j < n_ct
  const int cb = max(0, jb - n_ct_all);     // current tile = cb + (j - n_ct) for j >= n_ct
  const bool mass_only = p.mass_only != 0;
  const unsigned long long lim = p.wait_limit_ns;
  // Cached tiles are walked in order by every role: a CTile follows the
  // position (tile t, and for per-channel keys its chunk slot and key block)
  // with one division at the start, so the first token and the valid keys
  // of each tile cost no division (128-token tiles of the window, or the key
  // blocks of each chunk slot).
  struct CTile {
    int t, slot, blk;
  };
  auto ctile_at = [&](int t) -> CTile {
    CTile c{t, 0, 0};
    if (KCH) {
      c.slot = t / p.bpc;
      c.blk = t - c.slot * p.bpc;
    }
    return c;
  };
  auto ctile_next = [&](CTile& c) {
    ++c.t;
    if (KCH && ++c.blk == p.bpc) {
      c.blk = 0;
      ++c.slot;
    }
  };
  auto ctile_first = [&](const CTile& c) -> int {
    return KCH ? c.slot * p.chunk + c.blk * kBlockN : c.t * kBlockN;
  };
  auto ctile_count = [&](const CTile& c) -> int {
    if (!KCH) return min(kBlockN, p.n_s - c.t * kBlockN);
    return min(kBlockN, min(p.chunk, p.n_s - c.slot * p.chunk) - c.blk * kBlockN);
  };

  if (warp < C::kSoftmaxWarps) {
    // =========================== softmax ===========================
    const int q = warp >> 2;
    const int r = tid - q * 128;                      // row within the query tile
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    // every decision guarding a tcgen05 access is made warp-uniform: the
    // tensor-memory loads and stores are warp-collective
    bool ok = __all_sync(0xffffffffu, wait_bar(BAR(kBarQ), 0, lim, abort, p.status));
    {
      // group norms ||q'_g||^2 and group sums of the rotated query row
      float nrm[G], qsum[G];
#pragma unroll
      for (int g = 0; g < G; ++g) nrm[g] = qsum[g] = 0.f;
      const uint8_t* qt = smem + C::kQ + q * C::kTile;
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const int off = (c >> 3) * kHalf + sw128(r, c & 7);
        const uint4 v = *reinterpret_cast<const uint4*>(qt + off);
        uint4 vl = make_uint4(0u, 0u, 0u, 0u);
        if (PRECISE) vl = *reinterpret_cast<const uint4*>(qt + NQ * C::kTile + off);
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
      float cx[16], cz[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) cx[i] = cz[i] = 0.f;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float hi, lo;
        const int zc = PRECISE ? 3 * g : G + 3 * g;
        float(&zt)[16] = PRECISE ? cz : cx;
        split_h(kZeroQueryScale * qsum[g], hi, lo);
        zt[zc] = hi; zt[zc + 1] = hi; zt[zc + 2] = lo;
        if (PRECISE) {
          split_h(p.alpha_coef * nrm[g], hi, lo);
          cx[3 * g] = hi; cx[3 * g + 1] = hi; cx[3 * g + 2] = lo;
        } else {
          cx[g] = p.alpha_coef * nrm[g];
        }
      }
      write_ext_row(smem + C::kQx + q * C::kNExt * kExt, r, cx);
      if (PRECISE) write_ext_row(smem + C::kQx + q * C::kNExt * kExt + kExt, r, cz);
    }
    // exact correction: the row's rotated query (fp32) goes to tensor memory
    // for the per-channel terms; per group the maximum mu_g of q'_c^2 and the
    // series coefficients -log2(e) c_k M_k (pairs packed, two keys at a time).
    // Read from the query tile before the first QK can be issued (the tile is
    // overwritten once the cached QKs are done).
    constexpr int GE = EXACT ? G : 1;
    uint64_t mu2[GE], a2[GE][kFitTerms];
    const uint32_t t_q = tmem + C::kTQ + lane_off;
    if (EXACT) {
      const uint8_t* qt = smem + C::kQ + q * C::kTile;
      float mu[GE], mom[GE][kFitTerms];
#pragma unroll
      for (int g = 0; g < GE; ++g) {
        mu[g] = 0.f;
#pragma unroll
        for (int k = 0; k < kFitTerms; ++k) mom[g][k] = 0.f;
      }
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t v[32];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = 4 * cc + e;
          const int off = (c >> 3) * kHalf + sw128(r, c & 7);
          const uint4 hv = *reinterpret_cast<const uint4*>(qt + off);
          uint4 lv = make_uint4(0u, 0u, 0u, 0u);
          if (PRECISE) lv = *reinterpret_cast<const uint4*>(qt + NQ * C::kTile + off);
          const uint32_t w[4] = {hv.x, hv.y, hv.z, hv.w};
          const uint32_t wl[4] = {lv.x, lv.y, lv.z, lv.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            v[8 * e + 2 * i] = __float_as_uint(h_lo(w[i]) + h_lo(wl[i]));
            v[8 * e + 2 * i + 1] = __float_as_uint(h_hi(w[i]) + h_hi(wl[i]));
          }
        }
        ptx::tmem_st32(t_q + 32 * cc, v);
        const int g = (32 * cc) / GROUP;
#pragma unroll
        for (int k = 0; k < 32; ++k) mu[g] = fmaxf(mu[g], __uint_as_float(v[k]) * __uint_as_float(v[k]));
      }
      ptx::tmem_st_wait();
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t v[32];
        ptx::tmem_ld32(t_q + 32 * cc, v);
        const int g = (32 * cc) / GROUP;
        const float inv = mu[g] > 0.f ? 1.0f / mu[g] : 0.f;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float x = __uint_as_float(v[k]);
          const float u = x * x * inv;
          float pw = u;
          mom[g][0] += pw;
#pragma unroll
          for (int t = 1; t < kFitTerms; ++t) {
            pw *= u;
            mom[g][t] += pw;
          }
        }
      }
#pragma unroll
      for (int g = 0; g < GE; ++g) {
        mu2[g] = ptx::f2_pack(mu[g], mu[g]);
#pragma unroll
        for (int t = 0; t < kFitTerms; ++t) {
          const float a = -kLog2e * sinhc_fit(t) * mom[g][t];
          a2[g][t] = ptx::f2_pack(a, a);
        }
      }
    }
    ptx::fence_proxy_async_smem();
    ptx::mbar_arrive(BAR(kBarQx));

    float m = -INFINITY, l_s = 0.f, l_r = 0.f;
    const float sl2 = p.scale_log2;
    // per-channel keys: this row's column of the per-(row, tile) table
    const float* kch_row = KCH ? p.kch_c + (size_t)bh * n_ct_all * p.n_q + min(q0 + q * kBlockM + r, p.n_q - 1)
                               : nullptr;
    float toff_next = 0.f;
    if (KCH && n_ct > 0) toff_next = __ldg(kch_row + (size_t)kb * p.n_q);
    CTile sm_tile = ctile_at(kb);
    const uint32_t t_o = tmem + C::kTO + q * D + lane_off;
    for (int j = 0; j < n_t && ok; ++j) {
      const int b = NQ == 2 ? 0 : (j & 1);
      const uint32_t t_s = tmem + (q * C::kSBuf + b) * 128 + lane_off;
      const uint32_t par = NQ == 2 ? (j & 1) : ((j >> 1) & 1);
      if (!__all_sync(0xffffffffu, wait_bar(BAR(kBarS + q * C::kSBuf + b), par, lim, abort, p.status))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const int nv = j < n_ct ? ctile_count(sm_tile)
                              : min(kBlockN, p.n_r - (cb + j - n_ct) * kBlockN);
      if (j < n_ct) ctile_next(sm_tile);
      // per-channel keys: zero-point term minus correction of this row and
      // cached tile, one number (log2 units), folded into the exponent base;
      // the next tile's is fetched now, a tile ahead of its use
      float toff = 0.f;
      if (KCH && j < n_ct) {
        toff = toff_next;
        if (j + 1 < n_ct) toff_next = __ldg(kch_row + (size_t)(kb + j + 1) * p.n_q);
      }
      // One pass over the tile, 32 columns at a time, with the running base
      // m: P = 2^(s * scale * log2(e) - m).  The base only has to keep every
      // P inside the FP16 range, so it is raised only when a chunk's sum of
      // exponentials passes 2^15 (a bound on each of its terms); the chunk is
      // then recomputed from its scores, still in registers, against
      // max(m, chunk max), and the tile's earlier P chunks and sum are scaled
      // to the new base.  O and the running sums follow once per tile.
      const float m_in = m;
      const uint64_t sl2x2 = ptx::f2_pack(sl2, sl2);
      uint64_t acc = ptx::f2_pack(0.f, 0.f);
      // exact correction on cached tiles: (scale D_g / 2)^2 of the tile's keys
      // from the dequant warps, read after acquiring their writes through the
      // stage's V-half barrier (its phase for this tile has completed, and the
      // V half is not refilled before this tile's P is handed over and its PV
      // done); the series alone when every group of every key stays within
      // T <= kFitTmax
      const bool exact_tile = EXACT && j < n_ct;
      const float* dq =
          reinterpret_cast<const float*>(smem + C::kStages + (j & 1) * C::kStageBytes + C::kDsq);
      // bit c of `slow`: some row of the warp has, in 32-key chunk c, a key
      // with T > kFitTmax in some group (from the chunks' per-group maxima)
      uint32_t slow = 0u;
      if (exact_tile) {
        if (!__all_sync(0xffffffffu,
                        wait_bar(BAR(kBarFullV + (j & 1)), (j >> 1) & 1, lim, abort, p.status))) {
          ok = false;
          break;
        }
#pragma unroll
        for (int g = 0; g < GE; ++g) {
          const float4 tm = *reinterpret_cast<const float4*>(dq + 4 * kBlockN + 4 * g);
          float mu, unused;
          ptx::f2_unpack(mu2[g], mu, unused);
          slow |= (mu * tm.x > kFitTmax ? 1u : 0u) | (mu * tm.y > kFitTmax ? 2u : 0u) |
                  (mu * tm.z > kFitTmax ? 4u : 0u) | (mu * tm.w > kFitTmax ? 8u : 0u);
        }
        slow = __reduce_or_sync(0xffffffffu, slow);
      }
      // Full tiles take the chunk pass without column masks; only the last
      // tile of a segment (nv < 128 valid keys) masks its columns.
      auto chunk_pass = [&](auto masked_tag) {
        constexpr bool MASKED = decltype(masked_tag)::value;
#pragma unroll(EXACT ? 1 : 2)
        for (int c = 0; c < kBlockN / 32; ++c) {
          uint64_t nb[16];
          if (exact_tile) {   // before the scores are loaded: fewer live registers
            exact_series<GE>(dq + 32 * c, mu2, a2, nb);
            if ((slow >> c) & 1u) exact_fix<GE, D, GROUP>(dq + 32 * c, mu2, a2, t_q, nb);
          }
          uint32_t cur[32];
          ptx::tmem_ld32(t_s + 32 * c, cur);
          uint32_t pk[16];
          uint64_t cs = exact_tile ? exp_chunk_b<MASKED>(cur, nb, sl2x2, m, nv - 32 * c, pk)
                                   : exp_chunk<MASKED>(cur, sl2x2, m - toff, nv - 32 * c, pk);
          float cs_lo, cs_hi;
          ptx::f2_unpack(cs, cs_lo, cs_hi);
          // NaN-safe: an infinite or undefined sum also takes the slow path
          if (__any_sync(0xffffffffu, !(cs_lo + cs_hi <= kChunkSumLimit))) {
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            float cmax;
            if (exact_tile) {
#pragma unroll
              for (int k2 = 0; k2 < 16; ++k2) {
                float b0, b1;
                ptx::f2_unpack(nb[k2], b0, b1);
                const float x0 = fmaf(__uint_as_float(cur[2 * k2]), sl2, b0);
                const float x1 = fmaf(__uint_as_float(cur[2 * k2 + 1]), sl2, b1);
                const int i0 = (2 * k2) & 3, i1 = (2 * k2 + 1) & 3;
                m4[i0] = (!MASKED || 32 * c + 2 * k2 < nv) ? fmaxf(m4[i0], x0) : m4[i0];
                m4[i1] = (!MASKED || 32 * c + 2 * k2 + 1 < nv) ? fmaxf(m4[i1], x1) : m4[i1];
              }
              cmax = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            } else {
#pragma unroll
              for (int k = 0; k < 32; ++k)
                m4[k & 3] =
                    (!MASKED || 32 * c + k < nv) ? fmaxf(m4[k & 3], __uint_as_float(cur[k])) : m4[k & 3];
              cmax = fmaf(fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])), sl2, toff);
            }
            const float m_new = fmaxf(m, cmax);
            const float alpha = exp2f(m - m_new);   // 0 from the initial -inf base
            acc = ptx::f2_mul(acc, ptx::f2_pack(alpha, alpha));
            if (!mass_only && c > 0) {
              ptx::tmem_st_wait();
              for (int cc = 0; cc < c; ++cc) {
                uint32_t v[16];
                ptx::tmem_ld16(t_s + 16 * cc, v);
#pragma unroll
                for (int k = 0; k < 16; ++k) v[k] = ptx::f16x2_rn(h_lo(v[k]) * alpha, h_hi(v[k]) * alpha);
                ptx::tmem_st16(t_s + 16 * cc, v);
              }
            }
            m = m_new;
            cs = exact_tile ? exp_chunk_b<MASKED>(cur, nb, sl2x2, m, nv - 32 * c, pk)
                            : exp_chunk<MASKED>(cur, sl2x2, m - toff, nv - 32 * c, pk);
          }
          acc = ptx::f2_add(acc, cs);
          // P of columns [32c, 32c + 32) -> TMEM columns [16c, 16c + 16): all
          // of them already read
          if (!mass_only) ptx::tmem_st16(t_s + 16 * c, pk);
        }
      };
      if (nv < kBlockN) {
        chunk_pass(std::true_type{});
      } else {
        chunk_pass(std::false_type{});
      }
      if (NQ == 1 && j > 0) {
        // one-tile schedule: QK of this tile was issued before the previous
        // PV; O and the P-ready phases wait for that PV
        if (!__all_sync(0xffffffffu, wait_bar(BAR(kBarOStep), (j - 1) & 1, lim, abort, p.status))) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
      }
      if (__any_sync(0xffffffffu, m != m_in)) {
        const float alpha = exp2f(m_in - m);
        l_s *= alpha;
        l_r *= alpha;
        if (j > 0 && !mass_only) {
          const uint64_t a2 = ptx::f2_pack(alpha, alpha);
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32];
            ptx::tmem_ld32(t_o + 32 * c, v);
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
              float lo, hi;
              ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(v[k]), __uint_as_float(v[k + 1])), a2),
                             lo, hi);
              v[k] = __float_as_uint(lo);
              v[k + 1] = __float_as_uint(hi);
            }
            ptx::tmem_st32(t_o + 32 * c, v);
          }
        }
      }
      float sum_lo, sum_hi;
      ptx::f2_unpack(acc, sum_lo, sum_hi);
      const float sum = sum_lo + sum_hi;
      if (j < n_ct) l_s += sum; else l_r += sum;
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(BAR(kBarP + q));
    }

    // epilogue: O / (l_S + l_R), inverse rotation, BF16 store; masses
    const int row = q0 + q * kBlockM + r;
    if (ok) ok = wait_bar(BAR(kBarODone + q), 0, lim, abort, p.status);
    ok = __all_sync(0xffffffffu, ok && !*abort);
    if (ok && p.o_part != nullptr) {
      // key-range split: the unnormalized O' (rotated basis), the base and
      // both running sums of this range, for the merge kernel
      ptx::tc_fence_after();
      const bool store = row < p.n_q;
      const size_t base = ((size_t)blockIdx.z * gridDim.y + bh) * p.n_q + (store ? row : 0);
      if (!mass_only) {
        float4* dst = reinterpret_cast<float4*>(p.o_part + base * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          ptx::tmem_ld32(t_o + 32 * c, v);
          if (store) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[8 * c + e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                           __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
          }
        }
      }
      if (store) {
        p.st_part[base * 3] = m;
        p.st_part[base * 3 + 1] = l_s;
        p.st_part[base * 3 + 2] = l_r;
      }
    } else if (ok) {
      ptx::tc_fence_after();
      const float inv = 1.0f / (l_s + l_r);
      if (!mass_only) {
        // O = H^T O' = (1/sqrt(d)) diag(sigma) Sylvester(d) O', one row per
        // thread: butterflies h < 64 on each 64-column half in registers
        // (written back to TMEM), then h = 64 chunk by chunk
#pragma unroll
        for (int half = 0; half < D / 64; ++half) {
          float o[64];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t v[32];
            ptx::tmem_ld32(t_o + 64 * half + 32 * c, v);
#pragma unroll
            for (int k = 0; k < 32; ++k) o[32 * c + k] = __uint_as_float(v[k]) * inv;
          }
#pragma unroll
          for (int h = 1; h < 64; h <<= 1) {
#pragma unroll
            for (int i = 0; i < 64; ++i) {
              if ((i & h) == 0) {
                const float a = o[i], bb = o[i + h];
                o[i] = a + bb;
                o[i + h] = a - bb;
              }
            }
          }
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t v[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(o[32 * c + k]);
            ptx::tmem_st32(t_o + 64 * half + 32 * c, v);
          }
        }
        ptx::tmem_st_wait();
        // the tensor-memory loads are warp-collective: every lane takes part,
        // only the stores depend on the row being inside the chunk
        const bool store = row < p.n_q;
        uint16_t* dst = p.out + (static_cast<size_t>(bh) * p.n_q + (store ? row : 0)) * D;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t a[32], bq[32];
          ptx::tmem_ld32(t_o + 32 * c, a);
          if (D == 128) ptx::tmem_ld32(t_o + 64 + 32 * c, bq);
#pragma unroll
          for (int part = 0; part < (D == 128 ? 2 : 1); ++part) {
            const int ch_base = 64 * part + 32 * c;
            const uint32_t sw = p.sign_bits[ch_base >> 5];
            uint32_t pk[16];
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
              float v0, v1;
              if (D == 128) {
                v0 = part == 0 ? __uint_as_float(a[k]) + __uint_as_float(bq[k])
                               : __uint_as_float(a[k]) - __uint_as_float(bq[k]);
                v1 = part == 0 ? __uint_as_float(a[k + 1]) + __uint_as_float(bq[k + 1])
                               : __uint_as_float(a[k + 1]) - __uint_as_float(bq[k + 1]);
              } else {
                v0 = __uint_as_float(a[k]);
                v1 = __uint_as_float(a[k + 1]);
              }
              v0 *= ((sw >> k) & 1u) ? -p.inv_sqrt_d : p.inv_sqrt_d;
              v1 *= ((sw >> (k + 1)) & 1u) ? -p.inv_sqrt_d : p.inv_sqrt_d;
              pk[k >> 1] = pack_bf2(v0, v1);
            }
            if (store) {
#pragma unroll
              for (int e = 0; e < 4; ++e)
                *reinterpret_cast<uint4*>(dst + ch_base + 8 * e) =
                    make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
            }
          }
        }
      }
      if (row < p.n_q && p.p_s != nullptr) {
        p.p_s[static_cast<size_t>(bh) * p.n_q + row] = l_s * inv;
        p.p_r[static_cast<size_t>(bh) * p.n_q + row] = l_r * inv;
      }
    }
  } else if (warp < C::kMmaWarp) {
    // =========================== dequant ===========================
    const int r = tid - C::kDequantWarp * 32;
    const size_t head_tok = static_cast<size_t>(bh) * p.cap;
    // packed words of key r of tile j (zeros past the end of the window; the
    // tile at local index j is `pos`): the key half (codes, per-token steps,
    // or the per-channel block word of channel r) and the value half
    auto load_k = [&](int j, const CTile& pos, uint32_t (&kw)[NW], uint32_t (&ksz)[G],
                      uint32_t& kmeta) {
#pragma unroll
      for (int i = 0; i < NW; ++i) kw[i] = 0u;
#pragma unroll
      for (int g = 0; g < G; ++g) ksz[g] = 0u;
      kmeta = 0u;
      if (j >= n_ct) return;
      if constexpr (kCodesTma) {
        // tile j's key words, staged by the TMA thread (one tile at a time:
        // every dequant thread arrives once it has read its key's words)
        if (!wait_bar(BAR(kBarCodeK), j & 1, lim, abort, p.status)) return;
        if (r < ctile_count(pos)) {
          const uint4* kc = reinterpret_cast<const uint4*>(smem + C::kCodes + r * CB);
#pragma unroll
          for (int i = 0; i < NW / 4; ++i) {
            const uint4 v = kc[i];
            kw[4 * i] = v.x; kw[4 * i + 1] = v.y; kw[4 * i + 2] = v.z; kw[4 * i + 3] = v.w;
          }
          const uint4 z = *reinterpret_cast<const uint4*>(smem + C::kCodes + 128 * CB + r * 16);
          ksz[0] = z.x; ksz[1 % G] = z.y; ksz[2 % G] = z.z; ksz[3 % G] = z.w;
        }
        ptx::mbar_arrive(BAR(kBarCodeKFree));
        return;
      }
      // per-channel keys: thread r < D fetches the block's word of channel r
      if (KCH && r < D)
        kmeta = __ldg(p.k_sz + ((size_t)bh * p.kblk_per_head + pos.slot * p.bpc + pos.blk) * D + r);
      if (r >= ctile_count(pos)) return;
      if (!KVQ_IN_BOUNDS(ctile_first(pos) + r, p.cap, p.status, p.bounds_site)) return;
      const size_t tok = head_tok + (size_t)ctile_first(pos) + r;
      const uint4* kc = reinterpret_cast<const uint4*>(p.k_codes + tok * CB);
#pragma unroll
      for (int i = 0; i < NW / 4; ++i) {
        const uint4 v = __ldg(kc + i);
        kw[4 * i] = v.x; kw[4 * i + 1] = v.y; kw[4 * i + 2] = v.z; kw[4 * i + 3] = v.w;
      }
      if (!KCH) {
#pragma unroll
        for (int g = 0; g < G; ++g) ksz[g] = __ldg(p.k_sz + tok * G + g);
      }
    };
    auto load_v = [&](int j, const CTile& pos, uint32_t (&vw)[NW], uint32_t (&vsz)[G]) {
#pragma unroll
      for (int i = 0; i < NW; ++i) vw[i] = 0u;
#pragma unroll
      for (int g = 0; g < G; ++g) vsz[g] = 0u;
      if (j >= n_ct || mass_only) return;
      if constexpr (kCodesTma) {
        if (!wait_bar(BAR(kBarCodeV), j & 1, lim, abort, p.status)) return;
        if (r < ctile_count(pos)) {
          const uint8_t* vb = smem + C::kCodes + C::kCodeHalf;
          const uint4* vc = reinterpret_cast<const uint4*>(vb + r * CB);
#pragma unroll
          for (int i = 0; i < NW / 4; ++i) {
            const uint4 v = vc[i];
            vw[4 * i] = v.x; vw[4 * i + 1] = v.y; vw[4 * i + 2] = v.z; vw[4 * i + 3] = v.w;
          }
          const uint4 z = *reinterpret_cast<const uint4*>(vb + 128 * CB + r * 16);
          vsz[0] = z.x; vsz[1 % G] = z.y; vsz[2 % G] = z.z; vsz[3 % G] = z.w;
        }
        ptx::mbar_arrive(BAR(kBarCodeVFree));
        return;
      }
      if (r >= ctile_count(pos)) return;
      if (!KVQ_IN_BOUNDS(ctile_first(pos) + r, p.cap, p.status, p.bounds_site)) return;
      const size_t tok = head_tok + (size_t)ctile_first(pos) + r;
      const uint4* vc = reinterpret_cast<const uint4*>(p.v_codes + tok * CB);
#pragma unroll
      for (int i = 0; i < NW / 4; ++i) {
        const uint4 v = __ldg(vc + i);
        vw[4 * i] = v.x; vw[4 * i + 1] = v.y; vw[4 * i + 2] = v.z; vw[4 * i + 3] = v.w;
      }
#pragma unroll
      for (int g = 0; g < G; ++g) vsz[g] = __ldg(p.v_sz + tok * G + g);
    };
    uint32_t kw[NW], ksz[G], vw[NW], vsz[G], kmeta;
    // FP16 operand limits of the cached tiles (KVQ_ERR_RANGE when broken):
    // the key constant -(magic + o) D with magic <= 16 (which also keeps the
    // bias factor D^2 / 256 finite) and the value (code - z) D, at most
    // (|z| + 2^B - 1) D in magnitude
    constexpr float kKeyConst = 16.0f + (float)key_code_offset<BITS>();
    constexpr float kQmax = (float)((1 << BITS) - 1);
    bool range_bad = false;
    CTile dq_tile = ctile_at(kb), dq_next = dq_tile;
    ctile_next(dq_next);
    // per-thread loads: the next tile's words travel while the current tile
    // is written; staged words (kCodesTma): each half's words are read just
    // before waiting for that half of the stage, which releases the staging
    // buffer a tile ahead of the next copy
    if (!kCodesTma) {
      load_k(0, dq_tile, kw, ksz, kmeta);
      load_v(0, dq_tile, vw, vsz);
    }
    for (int j = 0; j < n_ct; ++j) {
      if (*abort) break;
      const int s = j & 1;
      const bool valid = r < ctile_count(dq_tile);
      uint8_t* st = smem + C::kStages + s * C::kStageBytes;
      // ---- K half: key rows and their extension rows ----
      // staged key words of this tile: read while the stage's K half is
      // still being released
      if (kCodesTma) load_k(j, dq_tile, kw, ksz, kmeta);
      if (j >= 2 && !wait_bar(BAR(kBarEmptyK + s), ((j >> 1) - 1) & 1, lim, abort, p.status)) break;
      if (KCH) {
        // the key block's per-channel steps and -magic * steps, shared
        // by the warpgroup through the stage's barrier (all 128 threads
        // arrive: a thread that writes here for tile j has waited on the
        // other stage's barrier for tile j - 1, so every thread is done
        // with this stage's previous tile)
        if (r < D) {
          range_bad |= !(bf16_lo(kmeta) * kKeyConst < kF16Max);
          const int k = BITS == 2 ? (r & 15) >> 1 : 0;
          reinterpret_cast<__half*>(st + C::kKch)[r] = __float2half_rn(bf16_lo(kmeta));
          reinterpret_cast<__half*>(st + C::kKch + 256)[r] =
              __float2half_rn(-(float)(pair_magic<BITS>(k) + key_code_offset<BITS>()) * bf16_lo(kmeta));
        }
        ptx::mbar_arrive(BAR(kBarKch + s));
        if (!wait_bar(BAR(kBarKch + s), (j >> 1) & 1, lim, abort, p.status)) break;
      }
      float cx[16], cz[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) cx[i] = cz[i] = 0.f;
      // exact correction: (scale D_g / 2)^2 of this key (0 past the window),
      // written with the V half
      float dsq[EXACT ? G : 1];
      if (EXACT) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float dt = p.half_scale * bf16_lo(ksz[g]);
          dsq[g] = dt * dt;
        }
      }
      if (valid && KCH) {
        dequant_row_kch<D, BITS>(kw, st + C::kKch, st + C::kKch + 256, st, r);
      } else if (valid) {
        dequant_row<D, BITS, GROUP, false>(kw, ksz, st, r);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float dl = bf16_lo(ksz[g]);
          range_bad |= !(dl * kKeyConst < kF16Max);
          float hi, lo;
          const int zc = PRECISE ? 3 * g : G + 3 * g;
          float(&zt)[16] = PRECISE ? cz : cx;
          split_h(((float)key_code_offset<BITS>() - bf16_hi(ksz[g])) * dl * kZeroKeyScale, hi, lo);
          zt[zc] = hi; zt[zc + 1] = lo; zt[zc + 2] = hi;
          if (PRECISE) {
            split_h(dl * dl * kBiasKeyScale, hi, lo);
            cx[3 * g] = hi; cx[3 * g + 1] = lo; cx[3 * g + 2] = hi;
          } else {
            cx[g] = dl * dl * kBiasKeyScale;
          }
        }
      } else {
        zero_row<D>(st, r);
      }
      write_ext_row(st + 2 * C::kTile, r, cx);
      if (PRECISE) write_ext_row(st + 2 * C::kTile + kExt, r, cz);
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(BAR(kBarFullK + s));
      // the next tile's key words travel while the V half is awaited and
      // written
      if (!kCodesTma) load_k(j + 1, dq_next, kw, ksz, kmeta);
      // ---- V half: value rows (and the exact correction's step terms) ----
      if (kCodesTma) load_v(j, dq_tile, vw, vsz);
      if (j >= 2 && !wait_bar(BAR(kBarEmptyV + s), ((j >> 1) - 1) & 1, lim, abort, p.status)) break;
      if (!mass_only) {
        if (valid) {
#pragma unroll
          for (int g = 0; g < G; ++g)
            range_bad |= !((fabsf(bf16_hi(vsz[g])) + kQmax) * bf16_lo(vsz[g]) < kF16Max);
          dequant_row<D, BITS, GROUP, true>(vw, vsz, st + C::kTile, r);
        } else {
          zero_row<D>(st + C::kTile, r);
        }
      }
      if (EXACT) {
        // per group the maximum over the warp's 32 keys as well
        float* dq = reinterpret_cast<float*>(st + C::kDsq);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float dt = dsq[g];
          dq[g * kBlockN + r] = dt;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) dt = fmaxf(dt, __shfl_xor_sync(0xffffffffu, dt, o));
          if ((r & 31) == 0) dq[4 * kBlockN + 4 * g + (r >> 5)] = dt;
        }
      }
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(BAR(kBarFullV + s));
      if (!kCodesTma) load_v(j + 1, dq_next, vw, vsz);
      dq_tile = dq_next;
      ctile_next(dq_next);
    }
    // a step size or value the FP16 tiles cannot carry: recorded, not fatal
    if (__any_sync(0xffffffffu, range_bad) && (r & 31) == 0) atomicCAS(p.status, 0, (int)KVQ_ERR_RANGE);
  } else if (warp == C::kMmaWarp) {
    // ============================= MMA =============================
    if (lane == 0) {
      constexpr uint32_t kIdS = ptx::idesc_f16kind(kBlockM, kBlockN, false, false);
      constexpr uint32_t kIdSbf = ptx::idesc_f16kind(kBlockM, kBlockN, false, true);
      constexpr uint32_t kIdO = ptx::idesc_f16kind(kBlockM, D, true, false);
      const uint32_t s_base = ptx::smem_u32(smem);
      bool ok = wait_bar(BAR(kBarQ), 0, lim, abort, p.status) && wait_bar(BAR(kBarQx), 0, lim, abort, p.status);
      if (ok && n_ct == 0) ptx::mbar_arrive(BAR(kBarQFree));
      bool q_orig_ready = false;

      auto wait_full = [&](int j) -> bool {
        const int s = j & 1;
        // cached tiles are uses 0, 1, ... of their stage's dequant barrier;
        // current tiles count only the TMA barrier's own uses of that stage
        const int use = j < n_ct ? (j >> 1) : (j >> 1) - ((n_ct + 1 - s) >> 1);
        if (!wait_bar(BAR(j < n_ct ? kBarFullK + s : kBarFullTma + s), use & 1, lim, abort, p.status))
          return false;
        if (j >= n_ct && !q_orig_ready) {
          if (!wait_bar(BAR(kBarQ), 1, lim, abort, p.status)) return false;
          q_orig_ready = true;
        }
        ptx::tc_fence_after();
        return true;
      };
      // the V half of a cached stage, before its first PV (current tiles
      // arrive whole through the TMA barrier awaited for their QK)
      auto wait_full_v = [&](int j) -> bool {
        if (j >= n_ct || mass_only) return true;
        if (!wait_bar(BAR(kBarFullV + (j & 1)), (j >> 1) & 1, lim, abort, p.status)) return false;
        ptx::tc_fence_after();
        return true;
      };
      // descriptors: built once, then advanced by (byte offset >> 4) in the
      // start-address field (the low 14 bits never carry: every operand lies
      // inside the 256 KB shared window)
      const uint64_t dsw = ptx::smem_desc(s_base, 16, 1024, ptx::kLayoutSw128);
      const uint64_t dvw = ptx::smem_desc(s_base, kHalf, 1024, ptx::kLayoutSw128);
      const uint64_t dex = ptx::smem_desc(s_base, 128, 256, ptx::kLayoutNone);
      auto at = [](uint64_t d, uint32_t off) { return d + (uint64_t)(off >> 4); };
      // per MMA only a 64-bit add of a compile-time step: operand bases are
      // turned into descriptors once per call
      auto issue_qk = [&](int j, int q, uint32_t d_tmem) {
        const uint32_t st = C::kStages + (j & 1) * C::kStageBytes;
        const uint32_t qa = C::kQ + q * C::kTile;
        const bool cached = j < n_ct;
        const uint32_t idq = cached ? kIdS : kIdSbf;
        const uint64_t da = at(dsw, qa), db = at(dsw, st);
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
          const uint64_t off = (uint64_t)(((s >> 2) * kHalf + (s & 3) * 32) >> 4);
          ptx::mma_f16(d_tmem, da + off, db + off, idq, s > 0);
        }
        if (cached) {
          if (PRECISE) {
            const uint64_t dl = at(dsw, qa + NQ * C::kTile);
#pragma unroll
            for (int s = 0; s < D / 16; ++s) {
              const uint64_t off = (uint64_t)(((s >> 2) * kHalf + (s & 3) * 32) >> 4);
              ptx::mma_f16(d_tmem, dl + off, db + off, kIdS, 1);
            }
          }
          // zero points and bias (its query columns are zero without the
          // correction); the precise layout spends a tile on each.  Per-
          // channel key tiles take both from the per-(row, tile) pre-pass,
          // in the softmax.
          if (!KCH) {
            const uint64_t dqx = at(dex, C::kQx + q * C::kNExt * kExt);
            const uint64_t dkx = at(dex, st + 2 * C::kTile);
            ptx::mma_f16(d_tmem, dqx, dkx, kIdS, 1);
            if (PRECISE) ptx::mma_f16(d_tmem, dqx + (kExt >> 4), dkx + (kExt >> 4), kIdS, 1);
          }
        }
      };
      auto issue_pv = [&](int j, int q, uint32_t p_tmem) {
        const uint64_t dv = at(dvw, C::kStages + (j & 1) * C::kStageBytes + C::kTile);
        const uint32_t o_tmem = tmem + C::kTO + q * D;
#pragma unroll
        for (int s = 0; s < kBlockN / 16; ++s) {
          ptx::mma_f16_ts(o_tmem, p_tmem + 8 * s, dv + (uint64_t)((s * 2048) >> 4), kIdO,
                          (j > 0 || s > 0) ? 1u : 0u);
        }
      };
      auto after_qk = [&](int j, int q) {   // query buffers free after the last cached QK
        if (j == n_ct - 1 && q == NQ - 1) ptx::mma_commit(BAR(kBarQFree));
      };

      if (ok && n_t > 0) {
        if (NQ == 2) {
          ok = wait_full(0);
          if (ok) {
            issue_qk(0, 0, tmem);
            ptx::mma_commit(BAR(kBarS + 0));
            issue_qk(0, 1, tmem + 128);
            ptx::mma_commit(BAR(kBarS + 1));
            ptx::mma_commit(BAR(kBarEmptyK + 0));
            after_qk(0, 1);
          }
          for (int j = 0; j < n_t && ok; ++j) {
            if (!(ok = wait_bar(BAR(kBarP + 0), j & 1, lim, abort, p.status))) break;
            ptx::tc_fence_after();
            if (!(ok = wait_full_v(j))) break;
            if (!mass_only) issue_pv(j, 0, tmem);
            const bool more = j + 1 < n_t;
            if (more) {
              if (!(ok = wait_full(j + 1))) break;
              issue_qk(j + 1, 0, tmem);
              ptx::mma_commit(BAR(kBarS + 0));
            }
            if (!(ok = wait_bar(BAR(kBarP + 1), j & 1, lim, abort, p.status))) break;
            ptx::tc_fence_after();
            if (!mass_only) issue_pv(j, 1, tmem + 128);
            ptx::mma_commit(BAR(kBarEmptyV + (j & 1)));
            if (more) {
              issue_qk(j + 1, 1, tmem + 128);
              ptx::mma_commit(BAR(kBarS + 1));
              ptx::mma_commit(BAR(kBarEmptyK + ((j + 1) & 1)));
              after_qk(j + 1, 1);
            }
          }
        } else {
          ok = wait_full(0);
          if (ok) {
            issue_qk(0, 0, tmem);
            ptx::mma_commit(BAR(kBarS + 0));
            ptx::mma_commit(BAR(kBarEmptyK + 0));
            after_qk(0, 0);
          }
          for (int j = 0; j < n_t && ok; ++j) {
            if (j + 1 < n_t) {
              if (!(ok = wait_full(j + 1))) break;
              issue_qk(j + 1, 0, tmem + ((j + 1) & 1) * 128);
              ptx::mma_commit(BAR(kBarS + ((j + 1) & 1)));
              ptx::mma_commit(BAR(kBarEmptyK + ((j + 1) & 1)));
              after_qk(j + 1, 0);
            }
            if (!(ok = wait_bar(BAR(kBarP + 0), j & 1, lim, abort, p.status))) break;
            ptx::tc_fence_after();
            if (!(ok = wait_full_v(j))) break;
            if (!mass_only) issue_pv(j, 0, tmem + (j & 1) * 128);
            // also in mass-only mode: keeps the softmax one tile behind
            ptx::mma_commit(BAR(kBarOStep));
            ptx::mma_commit(BAR(kBarEmptyV + (j & 1)));
          }
        }
      }
      // completion of every MMA issued: final O for the epilogues and a
      // drained tensor pipe before the tensor memory is released
      for (int q = 0; q < NQ; ++q) ptx::mma_commit(BAR(kBarODone + q));
      int drained = 0;
      wait_bar(BAR(kBarODone), 0, lim, &drained, p.status);
    }
    __syncwarp();
  } else {
    // ============================== TMA ==============================
    if (lane == 0) {
      const uint32_t s_base = ptx::smem_u32(smem);
      // a query tile starting past the last row is loaded from the last row
      // instead (its rows are computed but never stored): no box lies wholly
      // outside the tensor
      auto q_row = [&](int q) { return min(q0 + q * kBlockM, p.n_q - 1); };
      ptx::mbar_expect_tx(BAR(kBarQ), NQ * (PRECISE ? 2 : 1) * NKH * kHalf);
      for (int q = 0; q < NQ; ++q) {
        for (int h = 0; h < NKH; ++h) {
          ptx::tma_load_3d(s_base + C::kQ + q * C::kTile + h * kHalf, &tm_q, 64 * h, q_row(q), bh,
                           BAR(kBarQ));
          if (PRECISE)
            ptx::tma_load_3d(s_base + C::kQ + (NQ + q) * C::kTile + h * kHalf, &tm_qlo, 64 * h,
                             q_row(q), bh, BAR(kBarQ));
        }
      }
      // the cached tiles' packed words, one tile ahead of the dequant warps:
      // tile j's key (value) words once every dequant thread has read tile
      // j - 1's.  Bulk copies of count * 32 B of codes and count * 16 B of
      // (step, zero) words (16-byte aligned, multiples of 16 bytes)
      int last_ck = -1, last_cv = -1;
      if constexpr (kCodesTma) {
        auto stage_words = [&](int jj, const uint8_t* codes, const uint32_t* sz, uint32_t dst,
                               uint32_t bar) {
          const int t = kb + jj;
          const int cnt = min(kBlockN, p.n_s - t * kBlockN);
          // the tile's last token inside the head's slots (checked build);
          // on a failed check the copy still runs with nothing to move
          const bool in = KVQ_IN_BOUNDS(t * kBlockN + cnt - 1, p.cap, p.status, p.bounds_site);
          const size_t tok0 = (size_t)bh * p.cap + (size_t)t * kBlockN;
          if (!in) {
            ptx::mbar_arrive(bar);   // completes the phase without a copy
            return;
          }
          ptx::mbar_expect_tx(bar, (uint32_t)cnt * (CB + 16));
          ptx::bulk_load(dst, codes + tok0 * CB, (uint32_t)cnt * CB, bar);
          ptx::bulk_load(dst + 128 * CB, sz + tok0 * G, (uint32_t)cnt * 16, bar);
        };
        const uint32_t ck = s_base + C::kCodes, cv = ck + C::kCodeHalf;
        for (int jj = 0; jj < n_ct && !*abort; ++jj) {
          if (jj >= 1 && !wait_bar(BAR(kBarCodeKFree), (jj - 1) & 1, lim, abort, p.status)) break;
          stage_words(jj, p.k_codes, p.k_sz, ck, BAR(kBarCodeK));
          last_ck = jj;
          if (mass_only) continue;
          if (jj >= 1 && !wait_bar(BAR(kBarCodeVFree), (jj - 1) & 1, lim, abort, p.status)) break;
          stage_words(jj, p.v_codes, p.v_sz, cv, BAR(kBarCodeV));
          last_cv = jj;
        }
      }
      int last = -1;
      bool q_orig_issued = false;
      for (int j = n_ct; j < n_t; ++j) {
        if (*abort) break;
        const int s = j & 1;
        if (j == n_ct) {
          // the original BF16 queries replace the rotated ones once every
          // cached-tile QK MMA has completed
          if (!wait_bar(BAR(kBarQFree), 0, lim, abort, p.status)) break;
          ptx::mbar_expect_tx(BAR(kBarQ), NQ * NKH * kHalf);
          for (int q = 0; q < NQ; ++q)
            for (int h = 0; h < NKH; ++h)
              ptx::tma_load_3d(s_base + C::kQ + q * C::kTile + h * kHalf, &tm_qo, 64 * h,
                               q_row(q), bh, BAR(kBarQ));
          q_orig_issued = true;
        }
        // the V half's barrier: its commit follows the K half's, so both
        // halves of the stage are free
        if (j >= 2 && !wait_bar(BAR(kBarEmptyV + s), ((j >> 1) - 1) & 1, lim, abort, p.status)) break;
        const int key0 = (cb + j - n_ct) * kBlockN;
        const uint32_t st = s_base + C::kStages + s * C::kStageBytes;
        ptx::mbar_expect_tx(BAR(kBarFullTma + s), (mass_only ? 1 : 2) * NKH * kHalf);
        for (int h = 0; h < NKH; ++h) {
          ptx::tma_load_3d(st + h * kHalf, &tm_k, 64 * h, key0, bh, BAR(kBarFullTma + s));
          if (!mass_only)
            ptx::tma_load_3d(st + C::kTile + h * kHalf, &tm_v, 64 * h, key0, bh,
                             BAR(kBarFullTma + s));
        }
        last = j;
      }
      // on an abort, let the copies already issued land before the CTA exits
      if (*abort) {
        int ignore = 0;
        if (last_ck >= 0) wait_bar(BAR(kBarCodeK), last_ck & 1, lim, &ignore, p.status);
        if (last_cv >= 0) wait_bar(BAR(kBarCodeV), last_cv & 1, lim, &ignore, p.status);
        wait_bar(BAR(kBarQ), q_orig_issued ? 1 : 0, lim, &ignore, p.status);
        if (last >= 0) {
          const int s = last & 1;
          const int use = (last >> 1) - ((n_ct + 1 - s) >> 1);
          wait_bar(BAR(kBarFullTma + s), use & 1, lim, &ignore, p.status);
        }
      }
    }
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTCols);
  }
#undef BAR
}

// ---- key-range split: merge of the partial results -------------------------
//
// Every key range left its unnormalized O'_s (rotated basis), base m_s (log2
// units) and running sums l_S,s, l_R,s.  With m* = max_s m_s and
// w_s = 2^(m_s - m*):  O' = sum_s w_s O'_s / L, L = sum_s w_s (l_S,s + l_R,s),
// P_S = sum_s w_s l_S,s / L, P_R = sum_s w_s l_R,s / L -- the online-softmax
// combination of disjoint key sets -- then O = H^T O' (inverse rotation) to
// BF16.  A row is held by d/8 lanes, 8 channels each.
struct MergeArgs {
  const float* o_part;
  const float* st_part;
  int splits;
  long long rows;      // (B*H) * n_q
  uint16_t* out;
  float* p_s;
  float* p_r;
  uint32_t sign_bits[4];
  float inv_sqrt_d;
  int mass_only;
};

template <int D>
__global__ void __launch_bounds__(256) merge_splits_kernel(const MergeArgs a) {
  constexpr int LPR = D / 8;
  constexpr int RPW = 32 / LPR;
  const int lane = threadIdx.x & 31;
  const int t = lane % LPR;
  const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const int ch0 = 8 * t;
  // (selects, not a run-time index into the parameter array)
  const int wi = ch0 >> 5;
  const uint32_t sw = (wi == 0 ? a.sign_bits[0] : wi == 1 ? a.sign_bits[1]
                       : wi == 2 ? a.sign_bits[2] : a.sign_bits[3]) >> (ch0 & 31);
  for (long long r0 = warp0 * RPW; r0 < a.rows; r0 += nwarps * RPW) {
    const long long r = r0 + lane / LPR;
    const bool valid = r < a.rows;
    const long long rr = valid ? r : 0;
    // one pass over the ranges with a running base (loads of four ranges in
    // flight at a time)
    float mst = -INFINITY, ls = 0.f, lr = 0.f, o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = 0.f;
#pragma unroll 4
    for (int s = 0; s < a.splits; ++s) {
      const float* st = a.st_part + (s * a.rows + rr) * 3;
      const float ms = st[0], ss = st[1], sr = st[2];
      float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
      if (!a.mass_only) {
        const float4* src = reinterpret_cast<const float4*>(a.o_part + (s * a.rows + rr) * D + ch0);
        v0 = src[0];
        v1 = src[1];
      }
      const float mn = fmaxf(mst, ms);
      const float c_old = mst == -INFINITY ? 0.f : exp2f(mst - mn);
      const float w = ms == -INFINITY ? 0.f : exp2f(ms - mn);
      mst = mn;
      ls = fmaf(w, ss, ls * c_old);
      lr = fmaf(w, sr, lr * c_old);
      o[0] = fmaf(w, v0.x, o[0] * c_old); o[1] = fmaf(w, v0.y, o[1] * c_old);
      o[2] = fmaf(w, v0.z, o[2] * c_old); o[3] = fmaf(w, v0.w, o[3] * c_old);
      o[4] = fmaf(w, v1.x, o[4] * c_old); o[5] = fmaf(w, v1.y, o[5] * c_old);
      o[6] = fmaf(w, v1.z, o[6] * c_old); o[7] = fmaf(w, v1.w, o[7] * c_old);
    }
    const float inv = 1.0f / (ls + lr);
    if (!a.mass_only) {
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] *= inv;
      fwht_row<LPR>(o, t);   // all lanes: warp-collective shuffles
      uint32_t pk[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const float v0 = o[e] * (((sw >> e) & 1u) ? -a.inv_sqrt_d : a.inv_sqrt_d);
        const float v1 = o[e + 1] * (((sw >> (e + 1)) & 1u) ? -a.inv_sqrt_d : a.inv_sqrt_d);
        __nv_bfloat162 b = __floats2bfloat162_rn(v0, v1);
        pk[e / 2] = *reinterpret_cast<uint32_t*>(&b);
      }
      if (valid) *reinterpret_cast<uint4*>(a.out + r * D + ch0) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
    if (valid && t == 0 && a.p_s != nullptr) {
      a.p_s[r] = ls * inv;
      a.p_r[r] = lr * inv;
    }
  }
}

// ---- host side -------------------------------------------------------------

// the merge of a key-range split's partial results (one launch)
template <int D>
kvq_status launch_merge(const AttnLaunch& a, float inv_sqrt_d, cudaStream_t stream) {
  MergeArgs m;
  m.o_part = a.o_part;
  m.st_part = a.st_part;
  m.splits = a.splits;
  m.rows = (long long)a.bh * a.n_q;
  m.out = a.out;
  m.p_s = a.p_s;
  m.p_r = a.p_r;
  for (int i = 0; i < 4; ++i) m.sign_bits[i] = a.sign_bits[i];
  m.inv_sqrt_d = inv_sqrt_d;
  m.mass_only = a.mass_only;
  const long long warps = (m.rows + (32 / (D / 8)) - 1) / (32 / (D / 8));
  const unsigned blocks = (unsigned)((warps + 7) / 8);
  merge_splits_kernel<D><<<blocks, 256, 0, stream>>>(m);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

// One launch of the one-CTA kernel (the dispatcher launches the merge of a
// key-range split); select as in AttnParams.
template <int D, int BITS, int GROUP, int NQ, bool PRECISE, bool EXACT, bool KCH, bool STAGED = false>
kvq_status launch_t(const AttnLaunch& a, cudaStream_t stream, int select = 0) {
  using C = Cfg<D, NQ, PRECISE, EXACT, KCH,
                STAGED && codes_by_tma<D, BITS, GROUP, NQ, PRECISE, EXACT, KCH>()>;
  static std::atomic<uint64_t> limit_set{0};   // per template instance and device
  auto kern = attn_kernel<D, BITS, GROUP, NQ, PRECISE, EXACT, KCH, STAGED>;
  if (ensure_smem_limit(kern, C::kAlloc, limit_set) != cudaSuccess) return KVQ_ERR_CUDA;
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
  AttnParams p{};
  p.k_codes = a.k_codes;
  p.v_codes = a.v_codes;
  p.k_sz = a.k_sz;
  p.v_sz = a.v_sz;
  p.n_s = a.n_s;
  p.cap = a.cap;
  p.n_q = a.n_q;
  p.n_r = a.n_r;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.alpha_coef = a.corr == KVQ_CORR_TAYLOR ? -(a.scale / 24.0f) * 256.0f : 0.0f;
  p.half_scale = 0.5f * a.scale;
  p.corr = a.corr;
  p.mass_only = a.mass_only;
  p.out = a.out;
  p.p_s = a.p_s;
  p.p_r = a.p_r;
  for (int i = 0; i < 4; ++i) p.sign_bits[i] = a.sign_bits[i];
  p.inv_sqrt_d = (float)(1.0 / sqrt((double)D));
  p.wait_limit_ns = a.wait_limit_ns;
  const bool split = a.splits > 1;
  p.tiles_per_split = split ? a.tiles_per_split : (1 << 30);
  p.o_part = split ? a.o_part : nullptr;
  p.st_part = split ? a.st_part : nullptr;
  p.chunk = a.chunk;
  p.bpc = a.bpc;
  p.kblk_per_head = a.kblk_per_head;
  p.n_ct = a.n_ct;
  p.kch_c = a.kch_c;
  p.status = a.status;
  p.bounds_site = a.bounds_site;
  p.select = select;
  p.select_scale = a.scale * (1.0f / 4096.0f);
  p.qn2 = a.qn2;
  p.kn2 = a.kn2;
  dim3 grid((a.n_q + kBlockM * NQ - 1) / (kBlockM * NQ), a.bh, split ? a.splits : 1);
  kern<<<grid, C::kThreads, C::kAlloc, stream>>>(mq, mqlo, mqo, mk, mv, p);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace

}  // namespace kvq
