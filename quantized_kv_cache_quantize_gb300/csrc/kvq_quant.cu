// Quantize-append and rotation kernels (sm_103a).
//
// Quantize-append: for every new K and V row, rotate (randomized Hadamard,
// paper section 3), quantize per token and group with Eq. (1) (asymmetric
// round-to-nearest, step and zero point covering [min, max]) and pack the
// codes into the chunk slot of the sliding-window cache.
//
// Mapping: one thread per row (the whole row in registers, so the rotation
// needs no data exchange between threads); each warp owns tiles of 32 rows
// and stages the next tile into shared memory with asynchronous 16-byte
// copies while it quantizes the current one.  Codes leave in 16-byte
// stores, the (step, zero) records of a token in one store.  The kernel is
// bound by HBM bandwidth: per row it reads 2d bytes and writes
// d*bits/8 + 4*(d/group) bytes.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kvq_checks.cuh"
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

// Sign flips of the randomized rotation: word i of a BF16 row holds channels
// 2i (low half) and 2i + 1 (high half).  XOR with m[i] flips the sign bit of
// channel 2i + 1 (bit 31); channel 2i enters the first butterfly through an
// FMA by sl[i] = +-1 (an exact product, so the butterfly still rounds once).
struct PairSigns {
  uint32_t m[64];
  float sl[64];
};

// fl(x / d) from r = fl(1 / d): q0 = fl(x r), the exact residual x - q0 d by
// FMA, one correction step.  Correctly rounded while neither the residual
// nor the quotient leaves the normal range (Markstein's correction with a
// correctly rounded reciprocal).
__device__ __forceinline__ float div_step(float x, float d, float r) {
  const float q0 = __fmul_rn(x, r);
  return __fmaf_rn(__fmaf_rn(-q0, d, x), r, q0);
}

constexpr int kQWarps = 4;        // warps per block of the quantizer
constexpr int kQBlocksPerSm = 3;

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(ptx::smem_u32(smem_dst)),
               "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
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
template <int BITS, int N>
__device__ __forceinline__ uint32_t group_codes(float* xg, float mn, float mx, int& zfold) {
  const float qmax = float((1 << BITS) - 1);
  const QHdr h = group_header<BITS>(mn, mx);
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

// One row (one token's K or V row of one head), read from its warp's staged
// tile: d/8 16-byte chunks, chunk i of the tile's row `row` stored at
// 16 (i ^ (row mod d/8)) so that neither the copies nor the reads of a
// quarter-warp meet in a shared-memory bank.  fp32 butterflies in the order
// h = 1, 2, ..., d/2 (packed fp32 pairs from h = 2 on: each lane is the same
// correctly rounded add or subtract), per-group min/max, Eq. (1) codes,
// packed 16-byte stores.
template <int D, int BITS, int GROUP>
__device__ __forceinline__ void quantize_row(const QuantArgs& a, const PairSigns& sg,
                                             const uint8_t* tile, int row, unsigned r,
                                             unsigned per_kv) {
  constexpr int G = D / GROUP;
  constexpr int CODE_BYTES = D * BITS / 8;
  constexpr int PER_WORD = 32 / BITS;
  constexpr int CH = D / 8;

  const bool is_v = r >= per_kv;
  const unsigned rk = is_v ? r - per_kv : r;
  const unsigned bh = a.div_mul ? (__umulhi(rk, a.div_mul) >> a.div_shift) : (rk >> a.div_shift);
  const unsigned tok = rk - bh * (unsigned)a.n_new;

  const uint8_t* rowp = tile + row * (2 * D);
  float x[D];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) {
    const uint4 raw = *reinterpret_cast<const uint4*>(rowp + ((i ^ (row & (CH - 1))) << 4));
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[8 * i + 2 * k] = __uint_as_float(w[k] << 16);               // sign applied below
      x[8 * i + 2 * k + 1] = __uint_as_float((w[k] ^ sg.m[4 * i + k]) & 0xFFFF0000u);
    }
  }
  // butterflies: h = 1 on scalars (with the low channel's sign), then
  // packed pairs (x_i, x_i+1)
#pragma unroll
  for (int i = 0; i < D; i += 2) {
    const float u = x[i], v = x[i + 1];
    x[i] = __fmaf_rn(sg.sl[i / 2], u, v);
    x[i + 1] = __fmaf_rn(sg.sl[i / 2], u, -v);
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
  int zf[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float mn, mx;
    min_max<GROUP>(x + GROUP * g, mn, mx);
    rec[g] = group_codes<BITS, GROUP>(x + GROUP * g, mn, mx, zf[g]);
  }

  // pack: channel ch = 16w + 2k + h (INT2) / 8w + 2k + h (INT4) -> bits
  // BITS*k + 16h
  uint32_t words[D * BITS / 32];
#pragma unroll
  for (int w = 0; w < D * BITS / 32; ++w) words[w] = pack_word<BITS>(x + PER_WORD * w, zf[(PER_WORD * w) / GROUP]);

  if (!KVQ_IN_BOUNDS(a.first + tok, a.cap, a.status, a.bounds_site) ||
      !KVQ_IN_BOUNDS(bh, a.bh, a.status, a.bounds_site))
    return;
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

// Each warp walks tiles of 32 consecutive rows (the K rows of all (batch,
// head) pairs, then the V rows) with stride = all warps of the grid; the
// next tile is copied into the warp's other shared-memory stage (each copy
// instruction moves 32/(d/8) whole rows, 512 contiguous bytes) while the
// current one is quantized.
template <int D, int BITS, int GROUP>
__global__ void __launch_bounds__(kQWarps * 32, kQBlocksPerSm)
    quantize_rows_kernel(const QuantArgs a, const PairSigns sg) {
  constexpr int RB = 2 * D;          // bytes of one BF16 row
  constexpr int CH = D / 8;          // 16-byte chunks per row
  constexpr int RPI = 32 / CH;       // rows per copy instruction
  constexpr int TILE = 32 * RB;      // one warp's 32 rows
  extern __shared__ __align__(16) uint8_t qsm[];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  uint8_t* stage = qsm + wib * 2 * TILE;
  const unsigned per_kv = (unsigned)a.bh * (unsigned)a.n_new;   // < 2^30 (host check)
  const unsigned total = 2u * per_kv;
  const unsigned row_begin = a.v_only ? per_kv : 0u;              // V rows only
  const unsigned n_tiles = (total - row_begin + 31u) / 32u;
  const unsigned n_warps = gridDim.x * kQWarps;
  auto issue = [&](unsigned tile, uint8_t* dst) {
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      const int row = j * RPI + lane / CH, chunk = lane % CH;
      const unsigned r = row_begin + tile * 32u + (unsigned)row;
      if (r < total) {
        const bool is_v = r >= per_kv;
        const uint16_t* src = (is_v ? a.v_new : a.k_new) + (size_t)(is_v ? r - per_kv : r) * D + chunk * 8;
        cp_async16(dst + row * RB + ((chunk ^ (row & (CH - 1))) << 4), src);
      }
    }
    cp_async_commit();
  };
  unsigned tile = blockIdx.x * kQWarps + wib;
  if (tile < n_tiles) issue(tile, stage);
  for (int k = 0; tile < n_tiles; ++k, tile += n_warps) {
    const unsigned next = tile + n_warps;
    if (next < n_tiles) {
      issue(next, stage + ((k + 1) & 1) * TILE);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncwarp();
    const unsigned r = row_begin + tile * 32u + (unsigned)lane;
    if (r < total) quantize_row<D, BITS, GROUP>(a, sg, stage + (k & 1) * TILE, lane, r, per_kv);
    // every lane is done with this stage before the copy two tiles on
    __syncwarp();
  }
}

// ---- d = 128: each row split between the two warps of a pair ----------------
//
// Warp HF of a pair holds channels [64 HF, 64 HF + 64) of the pair's 32 rows
// (one row per lane), so a thread keeps 64 values instead of 128: half the
// registers and half the code per warp.  The butterflies h = 1 .. 32 stay
// inside a half; h = 64 pairs channel c with c + 64 across the two warps and
// goes through shared memory: HF = 0 keeps channels [0, 32) and sends
// [32, 64), HF = 1 keeps [96, 128) and sends [64, 96), so that afterwards
// HF = 0 owns channels [0, 32) and [64, 96), HF = 1 owns [32, 64) and
// [96, 128).  Groups of 32 channels then lie in one warp; groups of 64 swap
// their partial min / max once more.
//
// Both warps run one code path (one copy of the unrolled code in the
// instruction cache): warp 1 takes channels 96..127 with their signs flipped
// (an exact negation that every butterfly carries along), so its h = 32
// step leaves channels 96..127 in the first half of its registers, as warp 0
// has channels 0..31 there; both then keep their first half and send their
// second.  Warp 1's differences of the h = 64 step come out negated and take
// the scale -fl(1/sqrt(d)) (again exact).  Every value is the same fp32
// result as in the textbook order.
constexpr int kSplitWarps = 4;                  // two warp pairs per block
constexpr int kSplitBlocksPerSm = 4;
constexpr int kSplitStages = 3;
constexpr int kHalfRowBytes = 128;              // 64 BF16 channels
constexpr int kSplitTile = 32 * kHalfRowBytes;  // one warp's 32 half-rows
constexpr int kSplitSmem = kSplitWarps * (kSplitStages * kSplitTile + 32 * 4 * 4) + 64 * 4;

// named barrier of one warp pair (ids 1 and 2; 0 is __syncthreads)
__device__ __forceinline__ void pair_sync(int id) {
  asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
}

// 16-byte chunk i (0..7) of lane l's 128-byte slot, XOR-swizzled so that a
// quarter-warp's eight lanes use eight different bank groups
__device__ __forceinline__ int half_slot(int l, int i) { return l * kHalfRowBytes + ((i ^ (l & 7)) << 4); }

template <int BITS, int GROUP>
__device__ __forceinline__ void quantize_half_row(const QuantArgs& a, const uint32_t* msk,
                                                  uint8_t* own, const uint8_t* partner,
                                                  float* mm, const float* pmm, int lane, int HF,
                                                  unsigned rk, bool valid, bool is_v, int bar) {
  constexpr int H = 64, Q = 32;
  constexpr int G = 128 / GROUP;
  float x[H];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4 raw = *reinterpret_cast<const uint4*>(own + half_slot(lane, i));
    const uint4 mv = *reinterpret_cast<const uint4*>(msk + 4 * i);
    const uint32_t w[4] = {raw.x ^ mv.x, raw.y ^ mv.y, raw.z ^ mv.z, raw.w ^ mv.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int pl = 4 * i + k;
      const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xFFFF0000u);
      x[2 * pl] = __fadd_rn(lo, hi);          // h = 1
      x[2 * pl + 1] = __fsub_rn(lo, hi);
    }
  }
#pragma unroll
  for (int h = 2; h < H; h <<= 1) {
#pragma unroll
    for (int i = 0; i < H; i += 2) {
      if ((i & h) == 0) {
        const uint64_t A = ptx::f2_pack(x[i], x[i + 1]);
        const uint64_t B = ptx::f2_pack(x[i + h], x[i + h + 1]);
        ptx::f2_unpack(ptx::f2_add(A, B), x[i], x[i + 1]);
        ptx::f2_unpack(ptx::f2_sub(A, B), x[i + h], x[i + h + 1]);
      }
    }
  }
  // h = 64 across the pair.  Warp 1 took its channels 96..127 negated, so
  // its h = 32 butterflies left channels 96..127 (true values) in x[0..32)
  // and 64..95 in x[32..64): both warps keep x[0..32) (channels 32 HF ..
  // 32 HF + 31 before this step) and send x[32..64)
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 8; ++i)
    *reinterpret_cast<uint4*>(own + half_slot(lane, i)) =
        make_uint4(__float_as_uint(x[Q + 4 * i]), __float_as_uint(x[Q + 4 * i + 1]),
                   __float_as_uint(x[Q + 4 * i + 2]), __float_as_uint(x[Q + 4 * i + 3]));
  pair_sync(bar);
  // kept + received -> channel 32 HF + j; kept - received -> channel 64 +
  // 32 HF + j, negated in warp 1 (its kept values are the high channels):
  // the negation rides on the scale (exact)
  const uint64_t s2 = ptx::f2_pack(a.inv_sqrt_d, a.inv_sqrt_d);
  const float sd = HF ? -a.inv_sqrt_d : a.inv_sqrt_d;
  const uint64_t sd2 = ptx::f2_pack(sd, sd);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4 v = *reinterpret_cast<const uint4*>(partner + half_slot(lane, i));
    const float rv[4] = {__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                         __uint_as_float(v.w)};
#pragma unroll
    for (int e = 0; e < 4; e += 2) {
      const int j = 4 * i + e;
      const uint64_t kept = ptx::f2_pack(x[j], x[j + 1]);
      const uint64_t recv = ptx::f2_pack(rv[e], rv[e + 1]);
      ptx::f2_unpack(ptx::f2_mul(ptx::f2_add(kept, recv), s2), x[j], x[j + 1]);
      ptx::f2_unpack(ptx::f2_mul(ptx::f2_sub(kept, recv), sd2), x[Q + j], x[Q + j + 1]);
    }
  }
  uint32_t rec[2];
  int zf[2];
  if (GROUP == 32) {
    // x[0..32) is group HF, x[32..64) group 2 + HF
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      float mn, mx;
      min_max<Q>(x + Q * part, mn, mx);
      rec[part] = group_codes<BITS, Q>(x + Q * part, mn, mx, zf[part]);
    }
  } else {
    // x[0..32) is half of group 0, x[32..64) half of group 1
    float mn[2], mx[2];
#pragma unroll
    for (int part = 0; part < 2; ++part) min_max<Q>(x + Q * part, mn[part], mx[part]);
    *reinterpret_cast<float4*>(mm + 4 * lane) = make_float4(mn[0], mx[0], mn[1], mx[1]);
    pair_sync(bar);
    const float4 o = *reinterpret_cast<const float4*>(pmm + 4 * lane);
    mn[0] = fminf(mn[0], o.x);
    mx[0] = fmaxf(mx[0], o.y);
    mn[1] = fminf(mn[1], o.z);
    mx[1] = fmaxf(mx[1], o.w);
#pragma unroll
    for (int part = 0; part < 2; ++part)
      rec[part] = group_codes<BITS, Q>(x + Q * part, mn[part], mx[part], zf[part]);
  }
  if (!valid) return;
  const unsigned bh = a.div_mul ? (__umulhi(rk, a.div_mul) >> a.div_shift) : (rk >> a.div_shift);
  const unsigned tok = rk - bh * (unsigned)a.n_new;
  if (!KVQ_IN_BOUNDS(a.first + tok, a.cap, a.status, a.bounds_site) ||
      !KVQ_IN_BOUNDS(bh, a.bh, a.status, a.bounds_site))
    return;
  const size_t dst_tok = (size_t)bh * a.cap + a.first + tok;
  // codes: channels [32 HF, 32 HF + 32) and [64 + 32 HF, ...) -> bytes
  // [4 HF BITS, ...) and [8 BITS + 4 HF BITS, ...)
  constexpr int PER_WORD = 32 / BITS;
  constexpr int WPP = Q / PER_WORD;   // words per 32-channel part
  uint8_t* dc = (is_v ? a.v_codes : a.k_codes) + dst_tok * (128 * BITS / 8);
#pragma unroll
  for (int part = 0; part < 2; ++part) {
    uint32_t wd[WPP];
#pragma unroll
    for (int w = 0; w < WPP; ++w) wd[w] = pack_word<BITS>(x + Q * part + PER_WORD * w, zf[part]);
    uint8_t* d = dc + (part * 64 + HF * 32) * BITS / 8;
    if (WPP == 2) {
      *reinterpret_cast<uint2*>(d) = make_uint2(wd[0], wd[1 % WPP]);
    } else {
      *reinterpret_cast<uint4*>(d) = make_uint4(wd[0], wd[1 % WPP], wd[2 % WPP], wd[3 % WPP]);
    }
  }
  uint32_t* ds = (is_v ? a.v_sz : a.k_sz) + dst_tok * G;
  if (GROUP == 32) {
    ds[HF] = rec[0];
    ds[2 + HF] = rec[1];
  } else if (HF == 0) {
    *reinterpret_cast<uint2*>(ds) = make_uint2(rec[0], rec[1]);
  }
}

// Warp pairs walk tiles of 32 consecutive rows of one tensor (the K rows of
// all (batch, head) pairs in tiles [0, T), then the V rows in tiles [T, 2T))
// with stride = all pairs of the grid; each warp copies its half of the next
// tile (128-byte runs) into the next of its three shared-memory stages while
// it works on the current one.  Three stages because a stage slot also
// carries the h = 64 exchange: the copy into it waits until the partner has
// passed the following exchange.
template <int BITS, int GROUP>
__global__ void __launch_bounds__(kSplitWarps * 32, kSplitBlocksPerSm)
    quantize_split_kernel(const QuantArgs a, const PairSigns sg) {
  extern __shared__ __align__(16) uint8_t qsm[];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int hf = wib & 1;
  uint8_t* stages = qsm + wib * kSplitStages * kSplitTile;
  const uint8_t* pstages = qsm + (wib ^ 1) * kSplitStages * kSplitTile;
  float* mm_base = reinterpret_cast<float*>(qsm + kSplitWarps * kSplitStages * kSplitTile);
  float* mm = mm_base + wib * 128;
  const float* pmm = mm_base + (wib ^ 1) * 128;
  // sign masks of the two halves (bit 15: channel 2p, bit 31: channel 2p + 1
  // of pair p); the second half takes channels 96..127 negated as well
  uint32_t* msk_base = reinterpret_cast<uint32_t*>(mm_base + kSplitWarps * 128);
  if (threadIdx.x < 64) {
    const int p = threadIdx.x;   // pair of the row
    uint32_t m = sg.m[0];
#pragma unroll
    for (int q = 1; q < 64; ++q) m = q == p ? sg.m[q] : m;
    if (p >= 48) m ^= 0x80008000u;
    msk_base[p] = m;
  }
  __syncthreads();
  const uint32_t* msk = msk_base + 32 * hf;
  const unsigned per_kv = (unsigned)a.bh * (unsigned)a.n_new;   // < 2^30 (host check)
  const unsigned tiles_per = (per_kv + 31u) / 32u;
  const unsigned n_tiles = 2u * tiles_per;
  const unsigned n_pairs = gridDim.x * (kSplitWarps / 2);
  // this lane's share of a copy: rows 4j + lane / 8, chunk lane % 8
  const int crow = lane >> 3, cchunk = lane & 7;
  const int src_lane = crow * 128 + hf * 64 + cchunk * 8;   // BF16 elements
  const int dst_even = half_slot(crow, cchunk), dst_odd = half_slot(crow + 4, cchunk);
  auto issue = [&](unsigned tile, uint8_t* dst) {
    const bool v = tile >= tiles_per;
    const unsigned row0 = (v ? tile - tiles_per : tile) * 32u;
    const uint16_t* src = (v ? a.v_new : a.k_new) + (size_t)row0 * 128 + src_lane;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (row0 + 4u * j + (unsigned)crow < per_kv)
        cp_async16(dst + 512 * (j & ~1) + ((j & 1) ? dst_odd : dst_even), src + 512 * j);
    }
    cp_async_commit();
  };
  unsigned tile = (a.v_only ? tiles_per : 0u) + blockIdx.x * (kSplitWarps / 2) + (wib >> 1);
  if (tile < n_tiles) issue(tile, stages);
  int s = 0;
  for (int k = 0; tile < n_tiles; ++k, tile += n_pairs) {
    const unsigned next = tile + n_pairs;
    const int sn = s == kSplitStages - 1 ? 0 : s + 1;
    if (next < n_tiles) {
      issue(next, stages + sn * kSplitTile);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncwarp();
    const bool is_v = tile >= tiles_per;
    const unsigned rk = (is_v ? tile - tiles_per : tile) * 32u + (unsigned)lane;
    const bool valid = rk < per_kv;
    uint8_t* own = stages + s * kSplitTile;
    const uint8_t* par = pstages + s * kSplitTile;
    const int bar = 1 + (wib >> 1);
    quantize_half_row<BITS, GROUP>(a, msk, own, par, mm, pmm, lane, hf, rk, valid, is_v, bar);
    __syncwarp();
    s = sn;
  }
}

// ---- per-channel keys: Eq. (1) per channel over a block of tokens -----------
//
// One CTA of kKcThreads per (block of up to kKeyBlock tokens of the appended
// chunk, batch * head).
// 1. Rotation: LPR = d / 32 lanes per token row, 32 channels per lane,
//    butterflies h = 1 .. 16 in registers, the row written to shared memory,
//    read back transposed (lane j: channels {32u + (32 / LPR) j + v}), h = 32
//    (and 64) and the multiply by fl(1/sqrt(d)) in registers, written back in
//    place: the same fp32 operations in the same order as the per-token
//    kernels.  Rows are XOR-swizzled in 16-byte chunks (chunk c of lane jj's
//    channels at c ^ (2 jj + (t & 1)) for d = 128, c ^ (4 jj + (t & 3)) for
//    d = 64), which keeps a quarter-warp on eight bank groups.
// 2. Channel columns: kKcThreads / d threads per channel, each over a slice
//    of the tokens: min and max, combined through shared memory, the
//    channel's step and zero point (Eq. (1), the per-token group arithmetic),
//    then each value's code as a byte.
// 3. Token rows: two threads per token pack its codes into the cache's word
//    layout.
constexpr int kKcThreads = 256;

template <int D>
__device__ __forceinline__ int kc_swz(int jj, int t) {
  return D == 128 ? 2 * jj + (t & 1) : 4 * jj + (t & 3);
}

// float offset of channel c in a rotated row (token t)
template <int D>
__device__ __forceinline__ int kc_pos(int c, int t) {
  return 32 * (c >> 5) + 4 * (((c >> 2) & 7) ^ kc_swz<D>(c >> 5, t)) + (c & 3);
}

template <int D, int BITS>
__global__ void __launch_bounds__(kKcThreads) quantize_key_channels_kernel(const QuantArgs a) {
  constexpr int LPR = D / 32;                  // lanes per token row
  constexpr int VW = 32 / LPR;                 // channels per lane and run after the transpose
  constexpr int RPP = kKcThreads / LPR;        // rows per pass
  constexpr int P = kKcThreads / D;            // threads per channel column
  constexpr int SLICE = kKeyBlock / P;         // tokens per column thread
  constexpr int CB = D / 16;                   // 16-byte chunks of a code-byte row
  extern __shared__ __align__(16) uint8_t ksm[];
  float* rot = reinterpret_cast<float*>(ksm);                                   // [kKeyBlock][D]
  uint8_t* cb = ksm + kKeyBlock * D * 4;                                        // [kKeyBlock][D]
  float* mm = reinterpret_cast<float*>(cb + kKeyBlock * D);                     // [P][D][2]
  const int tid = threadIdx.x;
  const int blk = blockIdx.x;
  const int bh = blockIdx.y;
  const int t0 = blk * kKeyBlock;
  const int n = min(kKeyBlock, a.n_new - t0);

  // 1. rotation of the block's token rows
  {
    const int j = (tid & 31) % LPR;
    const uint32_t sw = j == 0 ? a.sign_bits[0] : j == 1 ? a.sign_bits[1] : j == 2 ? a.sign_bits[2]
                                                                                    : a.sign_bits[3];
    uint32_t z = 0;   // bit k: channel 2k of the lane's 32; bit 16 + k: channel 2k + 1
#pragma unroll
    for (int k = 0; k < 16; ++k) z |= (((sw >> (2 * k)) & 1u) << k) | (((sw >> (2 * k + 1)) & 1u) << (16 + k));
    // the lane's rows (kKeyBlock / RPP of them), all loaded before any is
    // transformed
    constexpr int NR = kKeyBlock / RPP;
    uint4 rawr[NR][4];
#pragma unroll
    for (int rr = 0; rr < NR; ++rr) {
      const int t = tid / LPR + rr * RPP;
      const bool live = t < n;
      const uint4* src = reinterpret_cast<const uint4*>(a.k_new + ((size_t)bh * a.n_new + t0 + (live ? t : 0)) * D + 32 * j);
#pragma unroll
      for (int k = 0; k < 4; ++k) rawr[rr][k] = live ? __ldg(src + k) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int rr = 0; rr < NR; ++rr) {   // the same rows count in every lane
      const int t = tid / LPR + rr * RPP;
      float* row = rot + t * D;
      const uint4 (&raw)[4] = rawr[rr];
      float x[32];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t u = w[i] ^ ((z << (15 - (4 * k + i))) & 0x80008000u);
          const float lo = __uint_as_float(u << 16), hi = __uint_as_float(u & 0xFFFF0000u);
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
      const int sj = kc_swz<D>(j, t);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4*>(row + 32 * j + 4 * (c ^ sj)) =
            make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]);
      __syncwarp();
      float y[32];
#pragma unroll
      for (int u = 0; u < LPR; ++u) {
        const int su = kc_swz<D>(u, t);
#pragma unroll
        for (int w4 = 0; w4 < VW / 4; ++w4) {
          const float4 v = *reinterpret_cast<const float4*>(row + 32 * u + 4 * (((VW / 4) * j + w4) ^ su));
          y[VW * u + 4 * w4] = v.x; y[VW * u + 4 * w4 + 1] = v.y;
          y[VW * u + 4 * w4 + 2] = v.z; y[VW * u + 4 * w4 + 3] = v.w;
        }
      }
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
      const uint64_t s2 = ptx::f2_pack(a.inv_sqrt_d, a.inv_sqrt_d);
#pragma unroll
      for (int i = 0; i < 32; i += 2) ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(y[i], y[i + 1]), s2), y[i], y[i + 1]);
      // back to the places read (each lane its own): the final rotated row
#pragma unroll
      for (int u = 0; u < LPR; ++u) {
        const int su = kc_swz<D>(u, t);
#pragma unroll
        for (int w4 = 0; w4 < VW / 4; ++w4)
          *reinterpret_cast<float4*>(row + 32 * u + 4 * (((VW / 4) * j + w4) ^ su)) =
              make_float4(y[VW * u + 4 * w4], y[VW * u + 4 * w4 + 1], y[VW * u + 4 * w4 + 2], y[VW * u + 4 * w4 + 3]);
      }
      __syncwarp();
    }
  }
  __syncthreads();

  // 2. channel columns: thread (part, c) takes tokens [part * SLICE, ...)
  const int c = tid % D;
  const int part = tid / D;
  const int ta = part * SLICE, tb = min(n, ta + SLICE);
  {
    // four independent running pairs (min and max are exact in any order)
    float mn[4] = {INFINITY, INFINITY, INFINITY, INFINITY};
    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 2
    for (int t = ta; t < tb; t += 4) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (t + u < tb) {
          const float v = rot[(t + u) * D + kc_pos<D>(c, t + u)];
          mn[u] = fminf(mn[u], v);
          mx[u] = fmaxf(mx[u], v);
        }
      }
    }
    mm[(part * D + c) * 2] = fminf(fminf(mn[0], mn[1]), fminf(mn[2], mn[3]));
    mm[(part * D + c) * 2 + 1] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
  }
  __syncthreads();
  {
    float mn = mm[2 * c], mx = mm[2 * c + 1];
#pragma unroll
    for (int p2 = 1; p2 < P; ++p2) {
      mn = fminf(mn, mm[(p2 * D + c) * 2]);
      mx = fmaxf(mx, mm[(p2 * D + c) * 2 + 1]);
    }
    const QHdr h = group_header<BITS>(mn, mx);
    if (part == 0 && KVQ_IN_BOUNDS(a.kblk_first + blk, a.kblk_per_head, a.status, a.bounds_site))
      a.k_sz[((size_t)bh * a.kblk_per_head + a.kblk_first + blk) * D + c] = h.rec;
#pragma unroll 8
    for (int t = ta; t < tb; ++t) {
      const float v = rot[t * D + kc_pos<D>(c, t)];
      cb[t * D + 16 * ((c >> 4) ^ (t & (CB - 1))) + (c & 15)] = (uint8_t)code_of_value<BITS>(v, h);
    }
  }
  __syncthreads();

  // 3. token t's codes into the packed words (two threads per token, half
  //    the words each): channel 16w + 2k + h (INT2) / 8w + 2k + h (INT4) at
  //    bits BITS*k + 16h of word w
  {
    constexpr int PER_WORD = 32 / BITS;
    constexpr int NW = D * BITS / 32;
    constexpr int NWH = NW / 2;             // words per thread
    constexpr int CH = NWH * PER_WORD / 16;  // 16-byte code chunks per thread
    const int t = tid >> 1, hw = tid & 1;
    if (t < n && KVQ_IN_BOUNDS(a.first + t0 + t, a.cap, a.status, a.bounds_site)) {
      uint32_t words[NWH];
#pragma unroll
      for (int w = 0; w < NWH; ++w) words[w] = 0u;
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        const int ci = hw * CH + i;   // code chunk of the row
        const uint4 v = *reinterpret_cast<const uint4*>(cb + t * D + 16 * (ci ^ (t & (CB - 1))));
        const uint32_t uu[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int ch = 16 * i + e;   // channel within this thread's half
          const uint32_t code = (uu[e >> 2] >> (8 * (e & 3))) & 0xFFu;
          const int jw = ch % PER_WORD;
          words[ch / PER_WORD] |= code << (BITS * (jw >> 1) + 16 * (jw & 1));
        }
      }
      uint8_t* drow = a.k_codes + ((size_t)bh * a.cap + a.first + t0 + t) * (D * BITS / 8) + hw * NWH * 4;
      if constexpr (NWH >= 4) {
#pragma unroll
        for (int i = 0; i < NWH / 4; ++i)
          reinterpret_cast<uint4*>(drow)[i] = make_uint4(words[4 * i], words[4 * i + 1], words[4 * i + 2], words[4 * i + 3]);
      } else {
        *reinterpret_cast<uint2*>(drow) = make_uint2(words[0], words[1 % NWH]);
      }
    }
  }
}

// Rotation of Q and V_R (FP16 out, with the FP16 remainder when asked) or of
// any BF16 rows (fp32 out).  LPR = d / 32 lanes per row, 32 channels per
// lane: lane j first holds channels [32j, 32j + 32) and runs the butterflies
// h = 1 .. 16 in registers; one transpose through shared memory then gives
// it channels {32u + (32 / LPR) j + v} (u < LPR, v < 32 / LPR), whose
// butterflies h = 32 (and 64) are again in registers.  Same fp32 operations
// in the same order as the textbook transform (h = 1, 2, ..., d/2, then the
// multiply by fl(1/sqrt(d))), so the fp32 output is bit for bit the
// quantizer's rotation.  Each lane's next row is loaded before the current
// one is transformed.
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
      if (a.out_f32) {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(dstp) + off);
#pragma unroll
        for (int q4 = 0; q4 < VW / 4; ++q4)
          dst[q4] = make_float4(y[VW * u + 4 * q4], y[VW * u + 4 * q4 + 1], y[VW * u + 4 * q4 + 2],
                                y[VW * u + 4 * q4 + 3]);
      } else {
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

template <int D, int BITS, int GROUP>
cudaError_t launch_q(const QuantArgs& a, cudaStream_t s) {
  PairSigns sg;
  for (int i = 0; i < 64; ++i) {
    const int c0 = 2 * i, c1 = 2 * i + 1;
    const uint32_t s0 = c0 < D ? (a.sign_bits[c0 >> 5] >> (c0 & 31)) & 1u : 0u;
    const uint32_t s1 = c1 < D ? (a.sign_bits[c1 >> 5] >> (c1 & 31)) & 1u : 0u;
    sg.m[i] = (s0 << 15) | (s1 << 31);
    sg.sl[i] = s0 ? -1.0f : 1.0f;
  }
  const long long rows = (a.v_only ? 1LL : 2LL) * a.bh * a.n_new;
  if (rows == 0) return cudaSuccess;
  const long long tiles = (rows + 31) / 32;
  if constexpr (D == 128) {
    const long long per = ((long long)a.bh * a.n_new + 31) / 32;   // tiles of one tensor
    const long long want = ((a.v_only ? per : 2 * per) + 1) / 2;
    const long long cap = (long long)sm_count() * kSplitBlocksPerSm;
    const unsigned blocks = (unsigned)(want < cap ? want : cap);
    static std::atomic<uint64_t> limit_set{0};   // per template instance and device
    const cudaError_t e = ensure_smem_limit(quantize_split_kernel<BITS, GROUP>, kSplitSmem, limit_set);
    if (e != cudaSuccess) return e;
    quantize_split_kernel<BITS, GROUP><<<blocks, kSplitWarps * 32, kSplitSmem, s>>>(a, sg);
    note_launch();
    return cudaGetLastError();
  } else {
    const long long want = (tiles + kQWarps - 1) / kQWarps;
    const long long cap = (long long)sm_count() * kQBlocksPerSm;
    const unsigned blocks = (unsigned)(want < cap ? want : cap);
    const int smem = kQWarps * 2 * 32 * 2 * D;
    static std::atomic<uint64_t> limit_set{0};   // per template instance and device
    const cudaError_t e = ensure_smem_limit(quantize_rows_kernel<D, BITS, GROUP>, smem, limit_set);
    if (e != cudaSuccess) return e;
    quantize_rows_kernel<D, BITS, GROUP><<<blocks, kQWarps * 32, smem, s>>>(a, sg);
    note_launch();
    return cudaGetLastError();
  }
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

namespace {

template <int D, int BITS>
cudaError_t launch_kc(const QuantArgs& a, cudaStream_t s) {
  if (a.n_new == 0 || a.bh == 0) return cudaSuccess;
  // fp32 rows + code bytes + per-part column min / max
  const int smem = kKeyBlock * D * 5 + (kKcThreads / D) * D * 2 * 4;
  static std::atomic<uint64_t> limit_set{0};   // per template instance and device
  const cudaError_t e = ensure_smem_limit(quantize_key_channels_kernel<D, BITS>, smem, limit_set);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)((a.n_new + kKeyBlock - 1) / kKeyBlock), (unsigned)a.bh);
  quantize_key_channels_kernel<D, BITS><<<grid, kKcThreads, smem, s>>>(a);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize_key_channels(const QuantArgs& a, int d, int bits, cudaStream_t stream,
                                         bool* supported) {
  *supported = true;
  if (d == 64 && bits == 2) return launch_kc<64, 2>(a, stream);
  if (d == 64 && bits == 4) return launch_kc<64, 4>(a, stream);
  if (d == 128 && bits == 2) return launch_kc<128, 2>(a, stream);
  if (d == 128 && bits == 4) return launch_kc<128, 4>(a, stream);
  *supported = false;
  return cudaSuccess;
}

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
