// Quantize-append with the rotation on the tensor cores (sm_103a): keys and
// values per token and group, keys per channel over 128-token blocks (the
// per-channel key mode), and the rotation alone (kvq_rotate's fp32 output).
//
// The randomized Hadamard rotation of a row (paper section 3, "Hadamard
// rotation") is the product x' = fl(1/sqrt(d)) * (W x) with the +-1 matrix
// W[n][k] = sigma_k (-1)^popcount(n & k) (Sylvester's matrix times the sign
// flips).  For a tile of 128 BF16 rows that is one chain of tcgen05 MMAs
// (M = 128 rows, N = d output channels, K = d input channels): every product
// x_k W[n][k] is exact, the tensor core sums the d products of a channel in
// fp32 and leaves the sums in tensor memory, one TMEM lane per row.  The
// epilogue warps read a row's sums, multiply by fl(1/sqrt(d)) and apply
// Eq. (1) per group (min/max, step, zero point, codes; the arithmetic of
// kvq_eq1.cuh), then store the packed codes and the (step, zero) records.
// The fp32 values differ from the butterfly order's by rounding only;
// kvq_rotate's fp32 output is exactly these values (the same kernel with
// the quantization left out), so the codes can be checked bit for bit.
//
// Why the tensor cores for an HBM-sized job: with the butterflies in fp32
// the per-token quantizer issues ~15 instructions per value and stays
// issue-bound well below the HBM rate; the MMA form moves the ~6 of them
// that the rotation costs onto the tensor pipe (a 128 x d x d product per
// tile, a few microseconds of tensor time for a whole chunk).
//
// Roles (one persistent CTA per SM, tiles of 128 rows dealt round-robin):
//   warp 0     one thread: TMA loads of a tile as d/64 boxes of
//              [128 rows][64 channels] (128-byte swizzle) into one of
//              kStages shared-memory stages;
//   warp 1     TMEM allocation; one thread issues a tile's d/16 MMAs into
//              one of kMqAcc accumulators and commits them to the stage's
//              "empty" and the accumulator's "full" barrier;
//   warps 2-17 the epilogue: warp w reads TMEM lanes 32 (w mod 4) .. + 31
//              (a rank of four warps covers a tile's 128 rows).  Per token:
//              each warp codes one group of those rows; the d / GROUP ranks
//              of a team share a tile, and the 4 GROUP / d teams take tiles
//              in turn.  Per channel (a tile is one 128-token block of one
//              head): warps 2-9 take the statistics (mq_kc_stats) and warps
//              10-17 the codes (mq_kc_codes) of consecutive tiles at once.
// Every mbarrier wait is bounded (the library's wait limit): when one runs
// out the kernel records KVQ_ERR_TIMEOUT, the other roles stop at their next
// wait, the TMA thread waits (bounded) for its copies in flight, the MMA
// thread for its last commit, and the TMEM is freed before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kvq_checks.cuh"
#include "kvq_eq1.cuh"
#include "kvq_internal.h"
#include "kvq_sm100.cuh"
#include "kvq_tmap.cuh"

namespace kvq {

namespace {

constexpr int kMqRows = 128;                       // rows per tile (the MMA's M)
static_assert(kMqRows == kKeyBlock, "a per-channel key block is one tile");
constexpr int kMqAcc = 4;                          // accumulators in tensor memory
constexpr int kMqRanks = 4;                        // epilogue warps per TMEM lane quarter
constexpr int kMqThreads = 64 + 128 * kMqRanks;    // TMA warp, MMA warp, epilogue

// what a launch computes
constexpr int kMqTokens = 0;        // per-token groups: codes and records (K and V rows)
constexpr int kMqRotOnly = 1;       // the fp32 rotation alone (kvq_rotate)
constexpr int kMqKeyChannels = 2;   // keys per channel over 128-token blocks

template <int D, int MODE>
struct MqCfg {
  static constexpr bool kKch = MODE == kMqKeyChannels;
  static constexpr int kStages = D == 64 ? 6 : kKch ? 3 : 4;
  static constexpr int kBox = kMqRows * 128;       // one [128][64] BF16 box (bytes)
  static constexpr int kTile = kBox * (D / 64);
  static constexpr int kWBox = D * 128;            // W: [D][64] per 64 input channels
  static constexpr int kWOff = kStages * kTile;
  // per-channel keys: the scaled tile [128 tokens][D] fp32, the column
  // passes' partial min / max [kKcParts][D][2] (kKcStatThreads threads), and
  // two buffers of channel headers (tile i in buffer i mod 2): per channel
  // (rcp, step, zero, flags) [D] float4; per channel pair (rcp, rcp', -step,
  // -step') [D / 2] float4 and (zero, zero') [D / 2] float2 for the packed
  // fp32 code pass; one flag per 32-channel chunk
  static constexpr int kKcStatThreads = 256;
  static constexpr int kKcParts = kKcStatThreads / D;
  static constexpr int kTOff = kWOff + kWBox * (D / 64);
  static constexpr int kMmOff = kTOff + (kKch ? kMqRows * D * 4 : 0);
  static constexpr int kHdrOff = kMmOff + (kKch ? kKcParts * D * 8 : 0);
  static constexpr int kHdrPair = D * 16;              // offsets inside a header buffer
  static constexpr int kHdrZero = kHdrPair + D * 8;
  static constexpr int kChunkFlag = kHdrZero + D * 4;
  static constexpr int kHdrBytes = kChunkFlag + 16;
  static constexpr int kBarOff = kKch ? kHdrOff + 2 * kHdrBytes : kHdrOff;
  static constexpr int kFull = 0;                  // [kStages] tile landed (TMA)
  static constexpr int kEmpty = kStages;           // [kStages] tile read by the MMAs
  static constexpr int kAccFull = 2 * kStages;     // [kMqAcc] accumulator written
  static constexpr int kAccEmpty = 2 * kStages + kMqAcc;   // [kMqAcc] read (its readers)
  static constexpr int kHdrFull = 2 * kStages + 2 * kMqAcc;   // [2] per-channel headers written
  static constexpr int kHdrEmpty = kHdrFull + 2;              // [2] headers used by the code warps
  static constexpr int kBars = 2 * kStages + 2 * kMqAcc + (kKch ? 4 : 0);
  static constexpr int kAbortOff = kBarOff + 8 * kBars;
  static constexpr int kTmemSlotOff = kAbortOff + 4;
  static constexpr int kSmem = kTmemSlotOff + 4 + 1024;   // + room to align the base
  static constexpr uint32_t kCols = kMqAcc * D;            // TMEM columns (256 or 512)
};

struct MqArgs {
  QuantArgs q;
  float* rot_out;      // rotation only: fp32 [rows][d]
  int rows;            // rows of one tensor (batch * heads * n_new)
  int tiles_k;         // tiles of the K rows (0 when only V is quantized)
  int tiles;           // all tiles (K tiles, then V tiles; per-channel keys:
                       // batch * heads * blocks, block-major within a head)
  int blocks;          // per-channel keys: 128-token blocks of the chunk
};

// Named barrier of the per-channel statistics warps (id 1, 256 threads; 0
// is __syncthreads), and the same barrier returning whether `v` held in
// every one of them.
__device__ __forceinline__ void stat_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ bool stat_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 256, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// Bounded wait on an mbarrier phase: false when the limit ran out (status
// and the CTA's abort flag set) or another role aborted.
__device__ bool mq_wait(uint32_t bar, uint32_t parity, unsigned long long limit_ns,
                        volatile int* abort, int* status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait_sleep(bar, parity, 20000u)) {
    if (*abort) return false;
    if (ptx::globaltimer() - t0 > limit_ns) {
      *abort = 1;
      if (status != nullptr) atomicCAS(status, 0, (int)KVQ_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// The same wait for work this thread issued itself, before the CTA exits:
// bounded, not cut short by the abort flag, and never shorter than
// kMinDrainNs (copies and MMAs in flight finish within microseconds; a tiny
// wait limit set by the caller must not let the CTA exit before them).
constexpr unsigned long long kMinDrainNs = 100000000ull;   // 100 ms
__device__ void mq_drain(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
  if (limit_ns < kMinDrainNs) limit_ns = kMinDrainNs;
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > limit_ns) return;
  }
}

// The bounded wait on a barrier nothing arrives on (kvq_selftest_wait_timeout):
// it runs out after limit_ns, records KVQ_ERR_TIMEOUT and returns.
__global__ void quant_wait_selftest_kernel(unsigned long long limit_ns, int* status) {
  __shared__ __align__(8) uint64_t b;
  __shared__ int abort_flag;
  const uint32_t a = ptx::smem_u32(&b);
  if (threadIdx.x == 0) {
    ptx::mbar_init(a, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  mq_wait(a, 0, limit_ns, &abort_flag, status);
}

// One group of one row (this thread's TMEM lane, channels [GROUP slot,
// GROUP slot + GROUP)): scale, Eq. (1), stores.  Warp-collective (the TMEM
// loads): every lane runs it, rows past the tensor's end (zero-filled by the
// TMA) store nothing.  At most 32 values are live: a group of 64 is read
// twice from tensor memory (min/max, then codes), by 32-channel chunks.
template <int D, int BITS, int GROUP, int MODE>
__device__ __forceinline__ void mq_group(const MqArgs& m, uint32_t taddr, int row, bool is_v,
                                         int slot) {
  const QuantArgs& a = m.q;
  constexpr int G = D / GROUP, NCH = GROUP / 32;
  constexpr int PER_WORD = 32 / BITS;
  constexpr int WPC = 32 / PER_WORD;   // code words per 32-channel chunk
  constexpr int CODE_BYTES = D * BITS / 8;
  const bool valid = row < m.rows;
  const uint64_t s2 = ptx::f2_pack(a.inv_sqrt_d, a.inv_sqrt_d);
  const int col0 = GROUP * slot;
  // channels [col, col + 32) of the row: the accumulator times fl(1/sqrt(d))
  auto load = [&](int col, float (&x)[32]) {
    uint32_t r[32];
    ptx::tmem_ld32(taddr + (uint32_t)col, r);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const uint64_t p = ptx::f2_pack(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
      ptx::f2_unpack(ptx::f2_mul(p, s2), x[j], x[j + 1]);
    }
  };
  if constexpr (MODE == kMqRotOnly) {
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      float x[32];
      load(col0 + 32 * c, x);
      if (valid) {
        float4* dst = reinterpret_cast<float4*>(m.rot_out + (size_t)row * D + col0 + 32 * c);
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[j] = make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
      }
    }
  } else {
    uint32_t words[NCH * WPC];
    float x[32];
    float mn, mx;
    load(col0, x);
    min_max<32>(x, mn, mx);
    if constexpr (NCH == 2) {
      float mn1, mx1;
      load(col0 + 32, x);
      min_max<32>(x, mn1, mx1);
      mn = fminf(mn, mn1);
      mx = fmaxf(mx, mx1);
    }
    const QHdr h = group_header<BITS>(mn, mx);
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      if constexpr (NCH == 2) load(col0 + 32 * c, x);
      int zf;
      apply_codes<BITS, 32>(x, h, zf);
#pragma unroll
      for (int w = 0; w < WPC; ++w) words[c * WPC + w] = pack_word<BITS>(x + PER_WORD * w, zf);
    }
    if (!valid) return;
    const unsigned rk = (unsigned)row;
    const unsigned bh = a.div_mul ? (__umulhi(rk, a.div_mul) >> a.div_shift) : (rk >> a.div_shift);
    const unsigned tok = rk - bh * (unsigned)a.n_new;
    if (!KVQ_IN_BOUNDS(a.first + tok, a.cap, a.status, a.bounds_site) ||
        !KVQ_IN_BOUNDS(bh, a.bh, a.status, a.bounds_site))
      return;
    const size_t dst_tok = (size_t)bh * a.cap + a.first + tok;
    // the group's code words: bytes [GROUP slot BITS / 8, + GROUP BITS / 8)
    uint8_t* dc = (is_v ? a.v_codes : a.k_codes) + dst_tok * CODE_BYTES + col0 * BITS / 8;
    if constexpr (NCH * WPC == 2) {
      *reinterpret_cast<uint2*>(dc) = make_uint2(words[0], words[1 % (NCH * WPC)]);
    } else {
#pragma unroll
      for (int i = 0; i < NCH * WPC / 4; ++i)
        reinterpret_cast<uint4*>(dc)[i] =
            make_uint4(words[4 * i], words[4 * i + 1], words[4 * i + 2], words[4 * i + 3]);
    }
    (is_v ? a.v_sz : a.k_sz)[dst_tok * G + slot] = h.rec;
  }
}

// The code of one value from its channel's header h = (rcp, step, zero,
// flags: 1 fast route, 2 clamp), as apply_codes does for a group: returns
// 1.5 * 2^23 + code (the zero point added, clamped when the channel needs
// it).
template <int BITS>
__device__ __forceinline__ float kc_code_one(float v, const float4 h) {
  constexpr float qmax = float((1 << BITS) - 1);
  const float kMagic = 12582912.0f;   // 1.5 * 2^23
  const uint32_t f = __float_as_uint(h.w);
  if (f & 1u) {
    const float q0 = __fmul_rn(v, h.x);
    const float q = __fmaf_rn(__fmaf_rn(-q0, h.y, v), h.x, q0);
    const float t = __fadd_rn(__fadd_rn(q, kMagic), h.z);
    return (f & 2u) ? fminf(fmaxf(t, kMagic), kMagic + qmax) : t;
  }
  // off the fast route: one IEEE division
  return __fadd_rn(fminf(fmaxf(__fadd_rn(rintf(__fdiv_rn(v, h.y)), h.z), 0.0f), qmax), kMagic);
}

// Per-channel keys: a tile is one 128-token block of one head.  Two roles of
// eight warps each work on consecutive tiles at once; warp (quarter,
// rank) covers tokens 32 quarter + lane and channels [64 rank, 64 rank + 64)
// (d = 64: [32 rank, 32 rank + 32)).
// Statistics warps (mq_kc_stats), tile i:
//   1. the accumulator times fl(1/sqrt(d)) into the shared tile
//      T[token][channel] (16-byte chunk cc of a row at cc ^ (token mod 8):
//      conflict-free row writes and column reads); they release their read
//      of the accumulator;
//   2. column passes: thread (part, c) takes channel c over 128 / P of the
//      block's tokens: min and max;
//   3. thread c (< d) combines the P partial results, computes the channel's
//      header (Eq. (1), group_header), stores the block's record and writes
//      the header into buffer i mod 2, once the code warps are done with
//      tile i - 2's.
// Code warps (mq_kc_codes), tile i once its headers are written: each warp
// reads its 32 tokens' channels from the accumulator again, codes them with
// the headers (broadcast reads; packed pairs when a chunk's channels all
// take the fast route, one value at a time otherwise), packs and stores them,
// and releases the accumulator and the header buffer.
template <int D, int BITS>
__device__ __forceinline__ bool mq_kc_stats(const MqArgs& m, uint8_t* sm, uint32_t tacc, int t, int i,
                                            int quarter, int rank, int lane, int tid_s,
                                            uint32_t acc_empty_bar, uint32_t hdr_full_bar,
                                            uint32_t hdr_empty_bar, unsigned long long lim,
                                            volatile int* abort_flag) {
  using C = MqCfg<D, kMqKeyChannels>;
  const QuantArgs& a = m.q;
  constexpr int NCH = D / 32;
  constexpr int CPW = NCH / 2;         // 32-channel chunks per warp
  constexpr int P = C::kKcParts;
  constexpr int SLICE = kMqRows / P;
  float* T = reinterpret_cast<float*>(sm + C::kTOff);
  float2* mm = reinterpret_cast<float2*>(sm + C::kMmOff);
  uint8_t* hb = sm + C::kHdrOff + (i & 1) * C::kHdrBytes;
  const int bh = t / m.blocks, blk = t - bh * m.blocks;
  const int nb = min(kMqRows, a.n_new - blk * kMqRows);
  const int tok = 32 * quarter + lane;
  {
    float* row = T + tok * D;
    const uint64_t s2 = ptx::f2_pack(a.inv_sqrt_d, a.inv_sqrt_d);
#pragma unroll 1
    for (int u = 0; u < CPW; ++u) {
      const int ch = CPW * rank + u;
      uint32_t r[32];
      ptx::tmem_ld32(tacc + (uint32_t)(32 * ch), r);
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        float y[4];
        ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(r[4 * cc]), __uint_as_float(r[4 * cc + 1])), s2),
                       y[0], y[1]);
        ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(r[4 * cc + 2]), __uint_as_float(r[4 * cc + 3])), s2),
                       y[2], y[3]);
        *reinterpret_cast<float4*>(row + 4 * ((8 * ch + cc) ^ (tok & 7))) = make_float4(y[0], y[1], y[2], y[3]);
      }
    }
  }
  ptx::tc_fence_before();
  __syncwarp();
  if (lane == 0) ptx::mbar_arrive(acc_empty_bar);
  stat_sync();
  {
    static_assert(SLICE % 8 == 0, "a column pass covers whole swizzle periods");
    const int c = tid_s % D, part = tid_s / D;
    const int ta = part * SLICE, tb = min(nb, ta + SLICE);
    // channel c of token k sits at k D + off[k mod 8]
    int off[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) off[u] = 4 * ((c >> 2) ^ u) + (c & 3);
    // four independent running pairs (min and max are exact in any order)
    float mn[4] = {INFINITY, INFINITY, INFINITY, INFINITY};
    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 2
    for (int tt = ta; tt < ta + SLICE; tt += 8) {
      const float* base = T + tt * D;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (tt + u < tb) {
          const float v = base[u * D + off[u]];
          mn[u & 3] = fminf(mn[u & 3], v);
          mx[u & 3] = fmaxf(mx[u & 3], v);
        }
      }
    }
    mm[part * D + c] = make_float2(fminf(fminf(mn[0], mn[1]), fminf(mn[2], mn[3])),
                                   fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])));
  }
  stat_sync();
  bool ok = true;
  if (tid_s < D) {
    const int c = tid_s;
    float mn = mm[c].x, mx = mm[c].y;
#pragma unroll
    for (int p2 = 1; p2 < P; ++p2) {
      mn = fminf(mn, mm[p2 * D + c].x);
      mx = fmaxf(mx, mm[p2 * D + c].y);
    }
    const QHdr h = group_header<BITS>(mn, mx);
    if (KVQ_IN_BOUNDS(a.kblk_first + blk, a.kblk_per_head, a.status, a.bounds_site) &&
        KVQ_IN_BOUNDS(bh, a.bh, a.status, a.bounds_site))
      a.k_sz[((size_t)bh * a.kblk_per_head + a.kblk_first + blk) * D + c] = h.rec;
    // the buffer held tile i - 2's headers: the code warps are done with it
    if (i >= 2) ok = mq_wait(hdr_empty_bar, ((i >> 1) - 1) & 1, lim, abort_flag, a.status);
    reinterpret_cast<float4*>(hb)[c] =
        make_float4(h.rcp, h.delta, h.zero, __uint_as_float((h.fast ? 1u : 0u) | (h.clamp ? 2u : 0u)));
    float* hp = reinterpret_cast<float*>(hb + C::kHdrPair) + 4 * (c >> 1) + (c & 1);
    hp[0] = h.rcp;
    hp[2] = -h.delta;
    reinterpret_cast<float*>(hb + C::kHdrZero)[c] = h.zero;
    // a chunk whose 32 channels all take the fast route (clamped or not:
    // the packed pass clamps every value, which changes nothing where no
    // code leaves [0, 2^B - 1])
    const bool simple = __all_sync(0xffffffffu, h.fast);
    if ((c & 31) == 0) reinterpret_cast<int*>(hb + C::kChunkFlag)[c >> 5] = simple ? 1 : 0;
    __threadfence_block();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(hdr_full_bar);
  }
  return ok;
}

template <int D, int BITS>
__device__ __forceinline__ void mq_kc_codes(const MqArgs& m, const uint8_t* sm, uint32_t tacc, int t,
                                            int i, int quarter, int rank, int lane) {
  using C = MqCfg<D, kMqKeyChannels>;
  const QuantArgs& a = m.q;
  constexpr int NCH = D / 32;
  constexpr int CPW = NCH / 2;
  constexpr int PER_WORD = 32 / BITS;
  constexpr int WPC = 32 / PER_WORD;   // code words per 32-channel chunk
  const uint8_t* hb = sm + C::kHdrOff + (i & 1) * C::kHdrBytes;
  const float4* hdr = reinterpret_cast<const float4*>(hb);
  const int bh = t / m.blocks, blk = t - bh * m.blocks;
  const int t0 = blk * kMqRows;
  const int nb = min(kMqRows, a.n_new - t0);
  const int tok = 32 * quarter + lane;
  const uint64_t s2 = ptx::f2_pack(a.inv_sqrt_d, a.inv_sqrt_d);
  const bool store = tok < nb && KVQ_IN_BOUNDS(a.first + t0 + tok, a.cap, a.status, a.bounds_site) &&
                     KVQ_IN_BOUNDS(bh, a.bh, a.status, a.bounds_site);
  uint8_t* drow = a.k_codes + ((size_t)bh * a.cap + a.first + t0 + tok) * (D * BITS / 8);
#pragma unroll 1
  for (int u = 0; u < CPW; ++u) {
    const int ch = CPW * rank + u;
    float x[32];
    {
      uint32_t r[32];
      ptx::tmem_ld32(tacc + (uint32_t)(32 * ch), r);
#pragma unroll
      for (int j = 0; j < 32; j += 2)
        ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), s2),
                       x[j], x[j + 1]);
    }
    if (reinterpret_cast<const int*>(hb + C::kChunkFlag)[ch]) {
      // every channel on the fast route: packed pairs, the headers in pair
      // layout (one 16-byte and one 8-byte broadcast load), every value
      // clamped to [1.5 * 2^23, 1.5 * 2^23 + 2^B - 1]
      const float4* hp = reinterpret_cast<const float4*>(hb + C::kHdrPair) + 16 * ch;
      const float2* hz = reinterpret_cast<const float2*>(hb + C::kHdrZero) + 16 * ch;
      const float kMagic = 12582912.0f;   // 1.5 * 2^23
      const float kTop = kMagic + float((1 << BITS) - 1);
      const uint64_t m2 = ptx::f2_pack(kMagic, kMagic);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float4 hq = hp[k];
        const float2 z = hz[k];
        const uint64_t xv = ptx::f2_pack(x[2 * k], x[2 * k + 1]);
        const uint64_t r2 = ptx::f2_pack(hq.x, hq.y);
        const uint64_t q0 = ptx::f2_mul(xv, r2);
        const uint64_t e = ptx::f2_fma(q0, ptx::f2_pack(hq.z, hq.w), xv);
        const uint64_t q = ptx::f2_fma(e, r2, q0);
        float c0, c1;
        ptx::f2_unpack(ptx::f2_add(ptx::f2_add(q, m2), ptx::f2_pack(z.x, z.y)), c0, c1);
        x[2 * k] = fminf(fmaxf(c0, kMagic), kTop);
        x[2 * k + 1] = fminf(fmaxf(c1, kMagic), kTop);
      }
    } else {
#pragma unroll 1
      for (int k = 0; k < 32; k += 2) {
        const float c0 = kc_code_one<BITS>(x[0], hdr[32 * ch + k]);
        const float c1 = kc_code_one<BITS>(x[1], hdr[32 * ch + k + 1]);
        // rotate the 32 values by two places (a rolled loop with
        // compile-time register indices): after 16 steps the codes are in
        // x[0..32) in channel order
#pragma unroll
        for (int j = 0; j < 30; ++j) x[j] = x[j + 2];
        x[30] = c0;
        x[31] = c1;
      }
    }
    uint32_t words[WPC];
#pragma unroll
    for (int w = 0; w < WPC; ++w) words[w] = pack_word<BITS>(x + PER_WORD * w, 0);
    if (store) {
      uint8_t* dc = drow + 32 * ch * BITS / 8;
      if constexpr (WPC == 2) {
        *reinterpret_cast<uint2*>(dc) = make_uint2(words[0], words[1 % WPC]);
      } else {
        *reinterpret_cast<uint4*>(dc) = make_uint4(words[0], words[1 % WPC], words[2 % WPC], words[3 % WPC]);
      }
    }
  }
}

template <int D, int BITS, int GROUP, int MODE>
__global__ void __launch_bounds__(kMqThreads, 1)
    quantize_mma_kernel(const __grid_constant__ CUtensorMap map_k,
                        const __grid_constant__ CUtensorMap map_v, const MqArgs m) {
  using C = MqCfg<D, MODE>;
  extern __shared__ uint8_t mq_raw[];
  // 128-byte swizzled operands: every box starts on a 1024-byte boundary
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(mq_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_u32(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kAbortOff);
  const uint32_t* tmem_slot = reinterpret_cast<const uint32_t*>(sm + C::kTmemSlotOff);
  const QuantArgs& a = m.q;
  const unsigned long long lim = a.wait_limit_ns;
  auto bar = [&](int i) { return sbase + C::kBarOff + 8 * i; };

  const int grid = (int)gridDim.x;
  // tile i of this CTA (t = blockIdx.x + i * grid) into stage i mod kStages
  auto issue = [&](int i, int t) {
    const int st = i % C::kStages;
    ptx::mbar_expect_tx(bar(C::kFull + st), C::kTile);
    if constexpr (MODE == kMqKeyChannels) {
      // block blk of head bh: tokens [128 blk, 128 blk + 128) of a [bh][n][d]
      // map (tokens past the chunk read as zeros)
      const int bh = t / m.blocks, blk = t - bh * m.blocks;
#pragma unroll
      for (int b = 0; b < D / 64; ++b)
        ptx::tma_load_3d(sbase + st * C::kTile + b * C::kBox, &map_k, 64 * b, blk * kMqRows, bh,
                         bar(C::kFull + st));
    } else {
      const bool v = t >= m.tiles_k;
      const int row0 = (v ? t - m.tiles_k : t) * kMqRows;
#pragma unroll
      for (int b = 0; b < D / 64; ++b)
        ptx::tma_load_2d(sbase + st * C::kTile + b * C::kBox, v ? &map_v : &map_k, 64 * b, row0,
                         bar(C::kFull + st));
    }
  };
  int issued = 0;   // thread 0: tiles whose loads are issued
  if (threadIdx.x == 0) {
    ptx::prefetch_tensormap(&map_k);
    ptx::prefetch_tensormap(&map_v);
    // an accumulator is released by the warps that read it: the 4 D / GROUP
    // warps of a team, or all 16 epilogue warps for per-channel keys (8
    // statistics and 8 code warps); a header buffer is written by the d / 32
    // warps that compute the headers and released by the 8 code warps
    constexpr uint32_t kReaders = MODE == kMqKeyChannels ? 4 * kMqRanks : 4 * (D / GROUP);
    for (int i = 0; i < C::kBars; ++i) {
      uint32_t count = 1u;
      if (i >= C::kAccEmpty && i < C::kAccEmpty + kMqAcc) count = kReaders;
      if (C::kKch && i >= C::kHdrFull && i < C::kHdrFull + 2) count = D / 32;
      if (C::kKch && i >= C::kHdrEmpty && i < C::kHdrEmpty + 2) count = 8u;
      ptx::mbar_init(bar(i), count);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
    // the inputs may come from the kernel launched before this one (a
    // programmatic dependent launch lets this prologue overlap its end)
    ptx::grid_dependency_wait();
    // the first kStages tiles need no free stage: their loads go out before
    // the operand matrix and the TMEM are set up
    for (int t = (int)blockIdx.x; t < m.tiles && issued < C::kStages; t += grid) issue(issued++, t);
  }
  // W in the B operand's layout: box b holds input channels [64 b, 64 b + 64)
  // of every output channel n (row n: 128 bytes, 16-byte chunk c at
  // c ^ (n mod 8)); entry (n, k) is BF16 +-1, negative when
  // popcount(n & k) + [sigma_k = -1] is odd
  for (int i = threadIdx.x; i < D * (D / 8); i += blockDim.x) {
    const int n = i / (D / 8), k0 = 8 * (i % (D / 8));
    const int wi = k0 >> 5;
    const uint32_t sw = wi == 0 ? a.sign_bits[0] : wi == 1 ? a.sign_bits[1]
                        : wi == 2 ? a.sign_bits[2] : a.sign_bits[3];
    uint32_t h[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const int k = k0 + e;
      const uint32_t s0 = ((uint32_t)__popc(n & k) ^ (sw >> (k & 31))) & 1u;
      const uint32_t s1 = ((uint32_t)__popc(n & (k + 1)) ^ (sw >> ((k + 1) & 31))) & 1u;
      h[e / 2] = (0x3F80u | (s0 << 15)) | ((0x3F80u | (s1 << 15)) << 16);
    }
    const int b = k0 >> 6, c = (k0 & 63) >> 3;
    *reinterpret_cast<uint4*>(sm + C::kWOff + b * C::kWBox + n * 128 + ((c ^ (n & 7)) << 4)) =
        make_uint4(h[0], h[1], h[2], h[3]);
  }
  ptx::fence_proxy_async_smem();
  if (warp == 1) {
    ptx::tmem_alloc(sbase + C::kTmemSlotOff, C::kCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // no global access before the previous kernel is complete (its reads of
  // the cache slot written here included)
  ptx::grid_dependency_wait();

  if (warp == 0) {
    if (lane == 0) {
      int i = issued;   // tiles whose loads were issued
      for (int t = (int)blockIdx.x + i * grid; t < m.tiles; t += grid, ++i) {
        const int s = i % C::kStages;
        if (!mq_wait(bar(C::kEmpty + s), ((i / C::kStages) - 1) & 1, lim, abort_flag, a.status))
          break;
        issue(i, t);
      }
      // the last loads of every stage have landed before the CTA moves on
      // (at once on the normal path: the MMAs waited for them)
      for (int j = i > C::kStages ? i - C::kStages : 0; j < i; ++j)
        mq_drain(bar(C::kFull + j % C::kStages), (j / C::kStages) & 1, lim);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_f16kind(kMqRows, D, false, true);
      int i = 0;   // tiles whose MMAs were issued
      for (int t = (int)blockIdx.x; t < m.tiles; t += grid, ++i) {
        const int s = i % C::kStages, ac = i % kMqAcc;
        if (!mq_wait(bar(C::kFull + s), (i / C::kStages) & 1, lim, abort_flag, a.status)) break;
        if (i >= kMqAcc &&
            !mq_wait(bar(C::kAccEmpty + ac), ((i / kMqAcc) - 1) & 1, lim, abort_flag, a.status))
          break;
        ptx::tc_fence_after();
        const uint32_t a0 = sbase + s * C::kTile, w0 = sbase + C::kWOff;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const int b = k >> 2, kk = k & 3;   // 64-channel box, 16-channel step in it
          const uint64_t da = ptx::smem_desc(a0 + b * C::kBox, 16, 1024, ptx::kLayoutSw128) + 2 * kk;
          const uint64_t dw = ptx::smem_desc(w0 + b * C::kWBox, 16, 1024, ptx::kLayoutSw128) + 2 * kk;
          ptx::mma_f16(tmem + (uint32_t)(ac * D), da, dw, idesc, k > 0 ? 1u : 0u);
        }
        ptx::mma_commit(bar(C::kEmpty + s));
        ptx::mma_commit(bar(C::kAccFull + ac));
      }
      // every MMA issued is complete before the TMEM is freed
      if (i > 0) mq_drain(bar(C::kAccFull + (i - 1) % kMqAcc), ((i - 1) / kMqAcc) & 1, lim);
    }
  } else if constexpr (MODE == kMqKeyChannels) {
    const int quarter = warp & 3;             // TMEM lanes 32 quarter .. + 31
    if (warp < 10) {
      // statistics warps 2-9
      const int rank = (warp - 2) >> 2;
      const int tid_s = (int)threadIdx.x - 64;
      bool ok = true;
      int i = 0;
      for (int t = (int)blockIdx.x; t < m.tiles; t += grid, ++i) {
        const int ac = i % kMqAcc;
        ok = ok && mq_wait(bar(C::kAccFull + ac), (i / kMqAcc) & 1, lim, abort_flag, a.status);
        // one decision for the whole role: its warps meet at named barriers
        if (!stat_all(ok)) break;
        ptx::tc_fence_after();
        ok = mq_kc_stats<D, BITS>(m, sm, tmem + (uint32_t)(ac * D) + ((uint32_t)(32 * quarter) << 16),
                                  t, i, quarter, rank, lane, tid_s, bar(C::kAccEmpty + ac),
                                  bar(C::kHdrFull + (i & 1)), bar(C::kHdrEmpty + (i & 1)), lim,
                                  abort_flag);
      }
    } else {
      // code warps 10-17
      const int rank = (warp - 10) >> 2;
      int i = 0;
      for (int t = (int)blockIdx.x; t < m.tiles; t += grid, ++i) {
        const int ac = i % kMqAcc;
        if (!__all_sync(0xffffffffu, mq_wait(bar(C::kHdrFull + (i & 1)), (i >> 1) & 1, lim,
                                              abort_flag, a.status)))
          break;
        // (complete already: the statistics warps waited for it) orders this
        // warp's tensor-memory reads after the MMAs
        if (!__all_sync(0xffffffffu, mq_wait(bar(C::kAccFull + ac), (i / kMqAcc) & 1, lim,
                                              abort_flag, a.status)))
          break;
        ptx::tc_fence_after();
        mq_kc_codes<D, BITS>(m, sm, tmem + (uint32_t)(ac * D) + ((uint32_t)(32 * quarter) << 16), t,
                             i, quarter, rank, lane);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(bar(C::kAccEmpty + ac));
          ptx::mbar_arrive(bar(C::kHdrEmpty + (i & 1)));
        }
      }
    }
  } else {
    // the four warps of a rank cover the four TMEM lane quarters; the ranks
    // split a tile's groups (D / GROUP of them, one rank each) and the
    // teams of ranks take tiles in turn
    constexpr int kSlots = D / GROUP;
    constexpr int kTeams = kMqRanks / kSlots;
    const int quarter = warp & 3;             // TMEM lanes 32 quarter .. + 31
    const int rank = (warp - 2) >> 2;
    const int team = rank / kSlots, slot = rank % kSlots;
    int i = team;
    for (int t = (int)blockIdx.x + team * grid; t < m.tiles; t += kTeams * grid, i += kTeams) {
      const int ac = i % kMqAcc;
      if (!__all_sync(0xffffffffu,
                      mq_wait(bar(C::kAccFull + ac), (i / kMqAcc) & 1, lim, abort_flag, a.status)))
        break;
      ptx::tc_fence_after();
      const bool v = t >= m.tiles_k;
      const int row = (v ? t - m.tiles_k : t) * kMqRows + 32 * quarter + lane;
      mq_group<D, BITS, GROUP, MODE>(
          m, tmem + (uint32_t)(ac * D) + ((uint32_t)(32 * quarter) << 16), row, v, slot);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(C::kAccEmpty + ac));
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kCols);
  }
}

int mq_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 1;
  return n;
}

template <int D, int BITS, int GROUP, int MODE>
cudaError_t launch_mq(const MqArgs& m, const CUtensorMap& mk, const CUtensorMap& mv,
                      cudaStream_t s) {
  using C = MqCfg<D, MODE>;
  if (m.tiles <= 0) return cudaSuccess;
  auto kern = quantize_mma_kernel<D, BITS, GROUP, MODE>;
  static std::atomic<uint64_t> limit_set{0};   // per template instance and device
  const cudaError_t e = ensure_smem_limit(kern, C::kSmem, limit_set);
  if (e != cudaSuccess) return e;
  const int sms = mq_sm_count();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(m.tiles < sms ? m.tiles : sms));
  cfg.blockDim = dim3(kMqThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  // programmatic dependent launch: the CTAs may start (prologue only) while
  // the previous kernel in the stream finishes; every global access waits
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t le = cudaLaunchKernelEx(&cfg, kern, mk, mv, m);
  note_launch();
  return le != cudaSuccess ? le : cudaGetLastError();
}

template <int D, int BITS, int GROUP>
cudaError_t launch_quant_t(const QuantArgs& a, cudaStream_t s) {
  MqArgs m{};
  m.q = a;
  m.rot_out = nullptr;
  m.rows = a.bh * a.n_new;
  const int per = (m.rows + kMqRows - 1) / kMqRows;
  m.tiles_k = a.v_only ? 0 : per;
  m.tiles = m.tiles_k + per;
  if (m.rows == 0) return cudaSuccess;
  CUtensorMap mk, mv;
  if (!make_rows_map(&mv, a.v_new, D, m.rows, kMqRows)) return cudaErrorInvalidValue;
  if (a.v_only) {
    mk = mv;
  } else if (!make_rows_map(&mk, a.k_new, D, m.rows, kMqRows)) {
    return cudaErrorInvalidValue;
  }
  return launch_mq<D, BITS, GROUP, kMqTokens>(m, mk, mv, s);
}

template <int D, int BITS>
cudaError_t launch_kc_t(const QuantArgs& a, cudaStream_t s) {
  if (a.n_new == 0 || a.bh == 0) return cudaSuccess;
  MqArgs m{};
  m.q = a;
  m.rot_out = nullptr;
  m.rows = a.n_new;
  m.blocks = (a.n_new + kMqRows - 1) / kMqRows;
  m.tiles = a.bh * m.blocks;
  m.tiles_k = m.tiles;
  CUtensorMap mk;
  if (!make_map(&mk, a.k_new, D, a.n_new, a.bh, true, kMqRows)) return cudaErrorInvalidValue;
  return launch_mq<D, BITS, 32, kMqKeyChannels>(m, mk, mk, s);
}

}  // namespace

cudaError_t launch_quantize_append_mma(const QuantArgs& a, int d, int bits, int group,
                                       cudaStream_t stream, bool* supported) {
  *supported = true;
#define KVQ_Q(D_, B_, G_) \
  if (d == D_ && bits == B_ && group == G_) return launch_quant_t<D_, B_, G_>(a, stream);
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

cudaError_t launch_quantize_key_channels_mma(const QuantArgs& a, int d, int bits,
                                             cudaStream_t stream, bool* supported) {
  *supported = true;
  if (d == 64 && bits == 2) return launch_kc_t<64, 2>(a, stream);
  if (d == 64 && bits == 4) return launch_kc_t<64, 4>(a, stream);
  if (d == 128 && bits == 2) return launch_kc_t<128, 2>(a, stream);
  if (d == 128 && bits == 4) return launch_kc_t<128, 4>(a, stream);
  *supported = false;
  return cudaSuccess;
}

cudaError_t launch_quant_wait_selftest(unsigned long long limit_ns, int* status,
                                      cudaStream_t stream) {
  quant_wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_rotate_mma_f32(const uint16_t* x, long long rows, int d,
                                  const uint32_t sign_bits[4], float* out, int* status,
                                  int* bounds_site, unsigned long long wait_limit_ns,
                                  cudaStream_t stream) {
  // segments of at most 2^30 rows (32-bit TMA row coordinates)
  constexpr long long kSeg = 1LL << 30;
  for (long long off = 0; off < rows; off += kSeg) {
    const long long n = rows - off < kSeg ? rows - off : kSeg;
    MqArgs m{};
    m.q.inv_sqrt_d = (float)(1.0 / sqrt((double)d));
    for (int i = 0; i < 4; ++i) m.q.sign_bits[i] = sign_bits[i];
    m.q.status = status;
    m.q.bounds_site = bounds_site;
    m.q.wait_limit_ns = wait_limit_ns;
    m.rot_out = out + off * d;
    m.rows = (int)n;
    m.tiles_k = (int)((n + kMqRows - 1) / kMqRows);
    m.tiles = m.tiles_k;
    CUtensorMap mk;
    if (!make_rows_map(&mk, x + off * d, d, n, kMqRows)) return cudaErrorInvalidValue;
    const cudaError_t e = d == 64 ? launch_mq<64, 2, 32, kMqRotOnly>(m, mk, mk, stream)
                                  : launch_mq<128, 2, 32, kMqRotOnly>(m, mk, mk, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace kvq
