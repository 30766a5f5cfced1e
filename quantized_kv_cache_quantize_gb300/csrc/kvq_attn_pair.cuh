// The corrected chunk attention on SM pairs (2-CTA clusters, tcgen05
// cta_group::2), head_dim 128, per-token keys, no correction or the Taylor
// term (the other modes run the one-CTA kernel of kvq_attn_kernel.cuh).
//
// Paper: "Quantized Keys Steal Attention" -- abstract and section 1 (the
// current chunk attends over the cached window and itself; the correction b
// is subtracted from cached-key scores only), Figure 3 caption (b), section 3
// (Eq. (1) dequantization, Hadamard rotation), Figure 2 caption (P_S, P_R).
// The arithmetic per score is the one-CTA kernel's; what changes is how the
// work of one key tile is shared by two SMs.
//
// One MMA of M = 256 rows spans both CTAs of a pair: rows 0-127 of A (the
// query tile) come from CTA 0's shared memory, rows 128-255 from CTA 1's,
// and B's N columns are split between them -- keys 0-63 of a key tile for
// the scores S = Q K^T, channels 0-63 / 64-127 of the value tile for
// O += P V.  So each CTA dequantizes half of every cached key tile: the K
// rows of 64 keys (two threads per key, 64 channels each) and 64 channels of
// all 128 value rows.  Per SM that is half the dequantization work of the
// one-CTA kernel for the same query rows, and half the K/V stage memory,
// which leaves room for the precise-query split (FP16 high and low query
// parts) with two query tiles per CTA.
//
// Roles per CTA (warps): softmax NQ warpgroups (own TMEM lanes, exactly as in
// the one-CTA kernel), dequant one warpgroup (its half of each cached tile),
// MMA one warp (CTA 0's issues every MMA of the pair; CTA 1's relays its
// CTA's TMA completions to CTA 0), TMA one warp (each CTA loads its own
// query rows and its half of each current-chunk tile).  Hand-offs:
//   to CTA 0's MMA thread: FullK / FullV (both dequant warpgroups, one
//     arrival per warp), P (both softmax warpgroups, one arrival per warp),
//     the local TMA barriers plus the peer's relayed ones;
//   from it, by multicast commits to both CTAs: S ready, K / V halves of a
//     stage free, query buffers free, PV done, all MMAs done.
// Every wait is bounded by the time limit; a wait that runs out sets the
// abort flag of both CTAs.  Both CTAs stay resident until the pair is done
// (cluster barrier before the tensor memory is released).
#pragma once

#include "kvq_attn_kernel.cuh"

namespace kvq {

namespace {

template <int NQ, bool PRECISE>
struct PairCfg {
  static constexpr int D = 128;
  static constexpr int kTileQ = kBlockM * D * 2;     // one query tile (two 64-channel sub-tiles)
  static constexpr int kKSub = 64 * 128;             // [64 keys][64 channels] FP16, swizzled
  static constexpr int kKTile = 2 * kKSub;           // this CTA's 64 keys x 128 channels
  static constexpr int kVTile = kBlockN * 64 * 2;    // 128 keys x this CTA's 64 channels
  static constexpr int kNExt = PRECISE ? 2 : 1;
  static constexpr int kExtK = 64 * 16 * 2;          // key-side extension rows of 64 keys
  static constexpr int kSBuf = NQ == 1 ? 2 : 1;
  static constexpr int kNS = 2;                      // K/V stages
  // shared memory
  static constexpr int kQ = 0;
  static constexpr int kQx = kQ + NQ * kTileQ * (PRECISE ? 2 : 1);
  static constexpr int kStages = ((kQx + NQ * kNExt * kExt) + 1023) / 1024 * 1024;
  static constexpr int kV = kKTile;                  // offsets inside a stage
  static constexpr int kKx = kKTile + kVTile;
  static constexpr int kStageBytes = kKTile + kVTile + kNExt * kExtK;
  static constexpr int kBar = kStages + kNS * kStageBytes;
  static constexpr int kBytes = kBar + 512;
  static constexpr int kAlloc = kBytes + 1024;
  // warps
  static constexpr int kSoftmaxWarps = 4 * NQ;
  static constexpr int kDequantWarp = kSoftmaxWarps;
  static constexpr int kMmaWarp = kSoftmaxWarps + 4;
  static constexpr int kThreads = (kSoftmaxWarps + 6) * 32;
  // tensor memory: S buffers, then the O tiles
  static constexpr int kTO = NQ * kSBuf * 128;
  static constexpr int kTCols = 512;
  static_assert(kTO + NQ * D <= kTCols, "tensor memory");
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
  static_assert(kAlloc <= 232448, "shared memory");
};

// mbarrier slots of the pair kernel ([n]: per stage / buffer / query tile).
// "leader" barriers are used in CTA 0 only, "local" ones in each CTA, "both"
// ones receive the multicast commits of CTA 0's MMA thread in both CTAs.
enum : int {
  kPbQ = 0,          // local: this CTA's query tiles landed (phase 0 rotated, 1 original)
  kPbQx = 1,         // local: query extension rows written (NQ * 128 arrivals)
  kPbQPeer = 2,      // leader: CTA 1's query tiles (and extension rows) ready (1 arrival)
  kPbQFree = 3,      // both: every cached-tile QK done, query buffers reusable
  kPbFullK = 4,      // leader [2]: K halves of a cached stage written (8 warp arrivals)
  kPbFullV = 6,      // leader [2]: V halves of a cached stage written (8 warp arrivals)
  kPbFullTma = 8,    // local [2]: this CTA's half of a current stage loaded
  kPbTmaPeer = 10,   // leader [2]: CTA 1's half of a current stage loaded (relayed)
  kPbEmptyK = 12,    // both [2]: K half of a stage consumed
  kPbEmptyV = 14,    // both [2]: V half of a stage consumed
  kPbS = 16,         // both [2]: S buffer ready
  kPbP = 18,         // leader [NQ]: P written in both CTAs (8 warp arrivals)
  kPbOStep = 20,     // both: PV of a tile done (one-tile schedule)
  kPbODone = 21,     // both [NQ]: every MMA done
  kPbCount = 23
};
constexpr int kPAbortOffset = kPbCount * 8;
constexpr int kPTmemSlotOffset = kPAbortOffset + 4;

// Bounded wait that acquires at cluster scope; when the limit runs out it
// records KVQ_ERR_TIMEOUT and raises the abort flag of this CTA and of the
// other CTA of the pair (peer_abort: its shared::cluster address).
__device__ bool wait_bar_pair(uint32_t bar, uint32_t parity, unsigned long long limit_ns,
                              volatile int* abort, int* status, uint32_t peer_abort) {
  if (ptx::mbar_try_wait_cl(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait_cl_sleep(bar, parity, 20000u)) {
    if (*abort) return false;
    if (ptx::globaltimer() - t0 > limit_ns) {
      *abort = 1;
      ptx::st_cluster_u32(peer_abort, 1u);
      atomicCAS(status, 0, (int)KVQ_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

template <int BITS, int GROUP, int NQ, bool PRECISE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PairCfg<NQ, PRECISE>::kThreads, 1)
    attn_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_qlo,
                     const __grid_constant__ CUtensorMap tm_qo,
                     const __grid_constant__ CUtensorMap tm_k64,
                     const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using C = PairCfg<NQ, PRECISE>;
  constexpr int D = 128;
  constexpr int G = D / GROUP;
  constexpr int GH = 64 / GROUP > 0 ? 64 / GROUP : 1;   // groups in 64 channels
  constexpr int CB = D * BITS / 8;       // packed bytes per token
  constexpr int NWH = CB / 8;            // packed words of 64 channels
  static_assert((PRECISE ? 3 : 4) * G <= 16, "extension columns");
  static_assert(GROUP <= 64, "a 64-channel half holds whole groups");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const int pair = blockIdx.x >> 1;
  const int bh = blockIdx.y;
  // a head the call gives to the one-CTA kernel: both CTAs of the pair leave
  // before anything is set up (no barrier, allocation or cluster access)
  if (head_not_mine(p, bh)) return;
  // query tile q of the pair: rows [pair_row0 + 256 q, + 256); this CTA's
  // 128 of them start at row_base(q)
  const int pair_row0 = pair * (2 * kBlockM * NQ);
  auto row_base = [&](int q) { return pair_row0 + 2 * kBlockM * q + kBlockM * (int)rank; };

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBar);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::kBar + kPAbortOffset);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kBar + kPTmemSlotOffset);
  const uint32_t bar0 = ptx::smem_u32(bars);
#define PB(i) (bar0 + 8u * (uint32_t)(i))
  // the same barrier in CTA 0 (shared::cluster address)
  const uint32_t lead_bar0 = ptx::mapa(bar0, 0);
#define LB(i) (lead_bar0 + 8u * (uint32_t)(i))
  const uint32_t peer_abort = ptx::mapa(ptx::smem_u32(const_cast<int*>(abort)), rank ^ 1u);

  if (tid == 0) {
    ptx::mbar_init(PB(kPbQ), 1);
    ptx::mbar_init(PB(kPbQx), NQ * 128);
    ptx::mbar_init(PB(kPbQPeer), 1);
    ptx::mbar_init(PB(kPbQFree), 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(PB(kPbFullK + s), 8);
      ptx::mbar_init(PB(kPbFullV + s), 8);
      ptx::mbar_init(PB(kPbFullTma + s), 1);
      ptx::mbar_init(PB(kPbTmaPeer + s), 1);
      ptx::mbar_init(PB(kPbEmptyK + s), 1);
      ptx::mbar_init(PB(kPbEmptyV + s), 1);
      ptx::mbar_init(PB(kPbS + s), 1);
      ptx::mbar_init(PB(kPbP + s), 8);
      ptx::mbar_init(PB(kPbODone + s), 1);
    }
    ptx::mbar_init(PB(kPbOStep), 1);
    *abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    // one warp of each CTA allocates the pair's tensor memory
    ptx::tmem_alloc2(ptx::smem_u32(tmem_slot), C::kTCols);
    ptx::tmem_relinquish2();
  }
  ptx::tc_fence_before();
  // barriers of both CTAs initialized before any arrival from the other
  ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int n_ct_all = (p.n_s + kBlockN - 1) / kBlockN;
  const int n_t_all = n_ct_all + (p.n_r + kBlockN - 1) / kBlockN;
  const int jb = blockIdx.z * p.tiles_per_split;
  const int je = min(n_t_all, jb + p.tiles_per_split);
  const int n_t = max(0, je - jb);
  const int n_ct = max(0, min(n_ct_all, je) - jb);
  const int kb = jb;
  const int cb = max(0, jb - n_ct_all);
  const bool mass_only = p.mass_only != 0;
  const unsigned long long lim = p.wait_limit_ns;
  constexpr int kNS = C::kNS;
  // uses of stage (j % kNS) by current tiles before tile j (TMA barriers)
  auto tma_use = [&](int j) { return j / kNS - (n_ct + kNS - 1 - j % kNS) / kNS; };
  auto wait = [&](uint32_t bar, uint32_t parity) {
    return wait_bar_pair(bar, parity, lim, abort, p.status, peer_abort);
  };

  if (warp < C::kSoftmaxWarps) {
    // =========================== softmax ===========================
    const int q = warp >> 2;
    const int r = tid - q * 128;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    bool ok = __all_sync(0xffffffffu, wait(PB(kPbQ), 0));
    {
      float nrm[G], qsum[G];
#pragma unroll
      for (int g = 0; g < G; ++g) nrm[g] = qsum[g] = 0.f;
      const uint8_t* qt = smem + C::kQ + q * C::kTileQ;
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const int off = (c >> 3) * kHalf + sw128(r, c & 7);
        const uint4 v = *reinterpret_cast<const uint4*>(qt + off);
        uint4 vl = make_uint4(0u, 0u, 0u, 0u);
        if (PRECISE) vl = *reinterpret_cast<const uint4*>(qt + NQ * C::kTileQ + off);
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
    ptx::fence_proxy_async_smem();
    ptx::mbar_arrive(PB(kPbQx));

    float m = -INFINITY, l_s = 0.f, l_r = 0.f;
    const float sl2 = p.scale_log2;
    const uint32_t t_o = tmem + C::kTO + q * D + lane_off;
    for (int j = 0; j < n_t && ok; ++j) {
      const int b = NQ == 2 ? 0 : (j & 1);
      const uint32_t t_s = tmem + (q * C::kSBuf + b) * 128 + lane_off;
      const uint32_t par = NQ == 2 ? (j & 1) : ((j >> 1) & 1);
      if (!__all_sync(0xffffffffu, wait(PB(kPbS + q * C::kSBuf + b), par))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const int nv = j < n_ct ? min(kBlockN, p.n_s - (kb + j) * kBlockN)
                              : min(kBlockN, p.n_r - (cb + j - n_ct) * kBlockN);
      const float m_in = m;
      const uint64_t sl2x2 = ptx::f2_pack(sl2, sl2);
      uint64_t acc = ptx::f2_pack(0.f, 0.f);
      // one pass over the tile, 32 columns at a time (as in the one-CTA
      // kernel: the base is raised only when a chunk's sum passes 2^15)
      auto chunk_pass = [&](auto masked_tag) {
        constexpr bool MASKED = decltype(masked_tag)::value;
#pragma unroll 2
        for (int c = 0; c < kBlockN / 32; ++c) {
          uint32_t cur[32];
          ptx::tmem_ld32(t_s + 32 * c, cur);
          uint32_t pk[16];
          uint64_t cs = exp_chunk<MASKED>(cur, sl2x2, m, nv - 32 * c, pk);
          float cs_lo, cs_hi;
          ptx::f2_unpack(cs, cs_lo, cs_hi);
          if (__any_sync(0xffffffffu, !(cs_lo + cs_hi <= kChunkSumLimit))) {
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int k = 0; k < 32; ++k)
              m4[k & 3] =
                  (!MASKED || 32 * c + k < nv) ? fmaxf(m4[k & 3], __uint_as_float(cur[k])) : m4[k & 3];
            const float cmax = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sl2;
            const float m_new = fmaxf(m, cmax);
            const float alpha = exp2f(m - m_new);
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
            cs = exp_chunk<MASKED>(cur, sl2x2, m, nv - 32 * c, pk);
          }
          acc = ptx::f2_add(acc, cs);
          if (!mass_only) ptx::tmem_st16(t_s + 16 * c, pk);
        }
      };
      if (nv < kBlockN) {
        chunk_pass(std::true_type{});
      } else {
        chunk_pass(std::false_type{});
      }
      if (NQ == 1 && j > 0) {
        if (!__all_sync(0xffffffffu, wait(PB(kPbOStep), (j - 1) & 1))) {
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
      // one arrival per warp on CTA 0's P barrier (the warp's tensor-memory
      // stores are complete: tcgen05.wait::st is warp-collective)
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(LB(kPbP + q));
    }

    // epilogue (this CTA's rows): as in the one-CTA kernel
    const int row = row_base(q) + r;
    if (ok) ok = wait(PB(kPbODone + q), 0);
    ok = __all_sync(0xffffffffu, ok && !*abort);
    if (ok && p.o_part != nullptr) {
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
        const bool store = row < p.n_q;
        uint16_t* dst = p.out + (static_cast<size_t>(bh) * p.n_q + (store ? row : 0)) * D;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t a[32], bq[32];
          ptx::tmem_ld32(t_o + 32 * c, a);
          ptx::tmem_ld32(t_o + 64 + 32 * c, bq);
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            const int ch_base = 64 * part + 32 * c;
            const uint32_t sw = p.sign_bits[ch_base >> 5];
            uint32_t pk[16];
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
              float v0 = part == 0 ? __uint_as_float(a[k]) + __uint_as_float(bq[k])
                                   : __uint_as_float(a[k]) - __uint_as_float(bq[k]);
              float v1 = part == 0 ? __uint_as_float(a[k + 1]) + __uint_as_float(bq[k + 1])
                                   : __uint_as_float(a[k + 1]) - __uint_as_float(bq[k + 1]);
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
    // K half: key kk = r / 2 of this CTA's 64 (tile keys 64 rank + kk),
    // channels [64 h, 64 h + 64), h = r % 2; the h = 0 thread also writes the
    // key's extension row.  V half: key r, channels [64 rank, 64 rank + 64).
    const int r = tid - C::kDequantWarp * 32;
    const int kk = r >> 1, kh = r & 1;
    const int kkey = 64 * (int)rank + kk;
    const size_t head_tok = static_cast<size_t>(bh) * p.cap;
    auto tile_count = [&](int j) { return min(kBlockN, p.n_s - (kb + j) * kBlockN); };
    auto load_k = [&](int j, uint32_t (&kw)[NWH], uint32_t (&ksz)[G]) {
#pragma unroll
      for (int i = 0; i < NWH; ++i) kw[i] = 0u;
#pragma unroll
      for (int g = 0; g < G; ++g) ksz[g] = 0u;
      if (j >= n_ct || kkey >= tile_count(j)) return;
      const size_t tok = head_tok + (size_t)(kb + j) * kBlockN + kkey;
      const uint4* kc = reinterpret_cast<const uint4*>(p.k_codes + tok * CB + kh * (CB / 2));
#pragma unroll
      for (int i = 0; i < NWH / 4; ++i) {
        const uint4 v = __ldg(kc + i);
        kw[4 * i] = v.x; kw[4 * i + 1] = v.y; kw[4 * i + 2] = v.z; kw[4 * i + 3] = v.w;
      }
#pragma unroll
      for (int g = 0; g < G; ++g) ksz[g] = __ldg(p.k_sz + tok * G + g);
    };
    auto load_v = [&](int j, uint32_t (&vw)[NWH], uint32_t (&vsz)[GH]) {
#pragma unroll
      for (int i = 0; i < NWH; ++i) vw[i] = 0u;
#pragma unroll
      for (int g = 0; g < GH; ++g) vsz[g] = 0u;
      if (j >= n_ct || mass_only || r >= tile_count(j)) return;
      const size_t tok = head_tok + (size_t)(kb + j) * kBlockN + r;
      const uint4* vc = reinterpret_cast<const uint4*>(p.v_codes + tok * CB + rank * (CB / 2));
#pragma unroll
      for (int i = 0; i < NWH / 4; ++i) {
        const uint4 v = __ldg(vc + i);
        vw[4 * i] = v.x; vw[4 * i + 1] = v.y; vw[4 * i + 2] = v.z; vw[4 * i + 3] = v.w;
      }
#pragma unroll
      for (int g = 0; g < GH; ++g) vsz[g] = __ldg(p.v_sz + tok * G + GH * rank + g);
    };
    uint32_t kw[NWH], ksz[G], vw[NWH], vsz[GH];
    constexpr float kKeyConst = 16.0f + (float)key_code_offset<BITS>();
    constexpr float kQmax = (float)((1 << BITS) - 1);
    bool range_bad = false;
    load_k(0, kw, ksz);
    load_v(0, vw, vsz);
    // every decision below is warp-uniform: the warps meet in __syncwarp
    // before their single arrival
    for (int j = 0; j < n_ct; ++j) {
      if (__any_sync(0xffffffffu, *abort)) break;
      const int s = j % kNS;
      const int use = j / kNS;
      uint8_t* st = smem + C::kStages + s * C::kStageBytes;
      // ---- K half ----
      if (j >= kNS && !__all_sync(0xffffffffu, wait(PB(kPbEmptyK + s), (use - 1) & 1))) break;
      const bool kvalid = kkey < tile_count(j);
      {
        // the groups of this thread's 64 channels
        uint32_t gsz[GH];
#pragma unroll
        for (int g = 0; g < GH; ++g) gsz[g] = kh ? ksz[GH + g] : ksz[g];
        if (kvalid) {
          dequant_row<64, BITS, GROUP, false>(kw, gsz, st + kh * C::kKSub, kk);
        } else {
          zero_row<64>(st + kh * C::kKSub, kk);
        }
      }
      if (kh == 0) {
        float cx[16], cz[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) cx[i] = cz[i] = 0.f;
        if (kvalid) {
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
        }
        write_ext_row(st + C::kKx, kk, cx);
        if (PRECISE) write_ext_row(st + C::kKx + C::kExtK, kk, cz);
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(LB(kPbFullK + s));
      load_k(j + 1, kw, ksz);
      // ---- V half ----
      if (j >= kNS && !__all_sync(0xffffffffu, wait(PB(kPbEmptyV + s), (use - 1) & 1))) break;
      if (!mass_only) {
        if (r < tile_count(j)) {
#pragma unroll
          for (int g = 0; g < GH; ++g)
            range_bad |= !((fabsf(bf16_hi(vsz[g])) + kQmax) * bf16_lo(vsz[g]) < kF16Max);
          dequant_row<64, BITS, GROUP, true>(vw, vsz, st + C::kV, r);
        } else {
          zero_row<64>(st + C::kV, r);
        }
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(LB(kPbFullV + s));
      load_v(j + 1, vw, vsz);
    }
    if (__any_sync(0xffffffffu, range_bad) && lane == 0) atomicCAS(p.status, 0, (int)KVQ_ERR_RANGE);
  } else if (warp == C::kMmaWarp) {
    // ============================= MMA =============================
    if (lane == 0 && rank == 0) {
      constexpr uint32_t kIdS = ptx::idesc_f16kind(2 * kBlockM, kBlockN, false, false);
      constexpr uint32_t kIdSbf = ptx::idesc_f16kind(2 * kBlockM, kBlockN, false, true);
      constexpr uint32_t kIdO = ptx::idesc_f16kind(2 * kBlockM, D, true, false);
      constexpr uint16_t kBoth = 3;
      const uint32_t s_base = ptx::smem_u32(smem);
      bool ok = wait(PB(kPbQ), 0) && wait(PB(kPbQx), 0) && wait(PB(kPbQPeer), 0);
      if (ok && n_ct == 0) ptx::mma_commit2_mc(PB(kPbQFree), kBoth);
      bool q_orig_ready = false;
      auto wait_full = [&](int j) -> bool {
        const int s = j % kNS;
        if (j < n_ct) {
          if (!wait(PB(kPbFullK + s), (j / kNS) & 1)) return false;
        } else {
          const int use = tma_use(j);
          if (!wait(PB(kPbFullTma + s), use & 1) || !wait(PB(kPbTmaPeer + s), use & 1)) return false;
          if (!q_orig_ready) {
            if (!wait(PB(kPbQ), 1) || !wait(PB(kPbQPeer), 1)) return false;
            q_orig_ready = true;
          }
        }
        ptx::tc_fence_after();
        return true;
      };
      auto wait_full_v = [&](int j) -> bool {
        if (j >= n_ct || mass_only) return true;
        if (!wait(PB(kPbFullV + j % kNS), (j / kNS) & 1)) return false;
        ptx::tc_fence_after();
        return true;
      };
      const uint64_t dsw = ptx::smem_desc(s_base, 16, 1024, ptx::kLayoutSw128);
      const uint64_t dvw = ptx::smem_desc(s_base, kHalf, 1024, ptx::kLayoutSw128);
      const uint64_t dex = ptx::smem_desc(s_base, 128, 256, ptx::kLayoutNone);
      auto at = [](uint64_t d, uint32_t off) { return d + (uint64_t)(off >> 4); };
      auto issue_qk = [&](int j, int q, uint32_t d_tmem) {
        const uint32_t st = C::kStages + (j % kNS) * C::kStageBytes;
        const uint32_t qa = C::kQ + q * C::kTileQ;
        const bool cached = j < n_ct;
        const uint32_t idq = cached ? kIdS : kIdSbf;
        const uint64_t da = at(dsw, qa), db = at(dsw, st);
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
          const uint64_t offa = (uint64_t)(((s >> 2) * kHalf + (s & 3) * 32) >> 4);
          const uint64_t offb = (uint64_t)(((s >> 2) * C::kKSub + (s & 3) * 32) >> 4);
          ptx::mma2_f16(d_tmem, da + offa, db + offb, idq, s > 0);
        }
        if (cached) {
          if (PRECISE) {
            const uint64_t dl = at(dsw, qa + NQ * C::kTileQ);
#pragma unroll
            for (int s = 0; s < D / 16; ++s) {
              const uint64_t offa = (uint64_t)(((s >> 2) * kHalf + (s & 3) * 32) >> 4);
              const uint64_t offb = (uint64_t)(((s >> 2) * C::kKSub + (s & 3) * 32) >> 4);
              ptx::mma2_f16(d_tmem, dl + offa, db + offb, kIdS, 1);
            }
          }
          const uint64_t dqx = at(dex, C::kQx + q * C::kNExt * kExt);
          const uint64_t dkx = at(dex, st + C::kKx);
          ptx::mma2_f16(d_tmem, dqx, dkx, kIdS, 1);
          if (PRECISE) ptx::mma2_f16(d_tmem, dqx + (kExt >> 4), dkx + (C::kExtK >> 4), kIdS, 1);
        }
      };
      auto issue_pv = [&](int j, int q, uint32_t p_tmem) {
        const uint64_t dv = at(dvw, C::kStages + (j % kNS) * C::kStageBytes + C::kV);
        const uint32_t o_tmem = tmem + C::kTO + q * D;
#pragma unroll
        for (int s = 0; s < kBlockN / 16; ++s)
          ptx::mma2_f16_ts(o_tmem, p_tmem + 8 * s, dv + (uint64_t)((s * 2048) >> 4), kIdO,
                           (j > 0 || s > 0) ? 1u : 0u);
      };
      auto after_qk = [&](int j, int q) {
        if (j == n_ct - 1 && q == NQ - 1) ptx::mma_commit2_mc(PB(kPbQFree), kBoth);
      };

      if (ok && n_t > 0) {
        if (NQ == 2) {
          ok = wait_full(0);
          if (ok) {
            issue_qk(0, 0, tmem);
            ptx::mma_commit2_mc(PB(kPbS + 0), kBoth);
            issue_qk(0, 1, tmem + 128);
            ptx::mma_commit2_mc(PB(kPbS + 1), kBoth);
            ptx::mma_commit2_mc(PB(kPbEmptyK + 0), kBoth);
            after_qk(0, 1);
          }
          for (int j = 0; j < n_t && ok; ++j) {
            if (!(ok = wait(PB(kPbP + 0), j & 1))) break;
            ptx::tc_fence_after();
            if (!(ok = wait_full_v(j))) break;
            if (!mass_only) issue_pv(j, 0, tmem);
            const bool more = j + 1 < n_t;
            if (more) {
              if (!(ok = wait_full(j + 1))) break;
              issue_qk(j + 1, 0, tmem);
              ptx::mma_commit2_mc(PB(kPbS + 0), kBoth);
            }
            if (!(ok = wait(PB(kPbP + 1), j & 1))) break;
            ptx::tc_fence_after();
            if (!mass_only) issue_pv(j, 1, tmem + 128);
            ptx::mma_commit2_mc(PB(kPbEmptyV + j % kNS), kBoth);
            if (more) {
              issue_qk(j + 1, 1, tmem + 128);
              ptx::mma_commit2_mc(PB(kPbS + 1), kBoth);
              ptx::mma_commit2_mc(PB(kPbEmptyK + (j + 1) % kNS), kBoth);
              after_qk(j + 1, 1);
            }
          }
        } else {
          ok = wait_full(0);
          if (ok) {
            issue_qk(0, 0, tmem);
            ptx::mma_commit2_mc(PB(kPbS + 0), kBoth);
            ptx::mma_commit2_mc(PB(kPbEmptyK + 0), kBoth);
            after_qk(0, 0);
          }
          for (int j = 0; j < n_t && ok; ++j) {
            if (j + 1 < n_t) {
              if (!(ok = wait_full(j + 1))) break;
              issue_qk(j + 1, 0, tmem + ((j + 1) & 1) * 128);
              ptx::mma_commit2_mc(PB(kPbS + ((j + 1) & 1)), kBoth);
              ptx::mma_commit2_mc(PB(kPbEmptyK + (j + 1) % kNS), kBoth);
              after_qk(j + 1, 0);
            }
            if (!(ok = wait(PB(kPbP + 0), j & 1))) break;
            ptx::tc_fence_after();
            if (!(ok = wait_full_v(j))) break;
            if (!mass_only) issue_pv(j, 0, tmem + (j & 1) * 128);
            ptx::mma_commit2_mc(PB(kPbOStep), kBoth);
            ptx::mma_commit2_mc(PB(kPbEmptyV + j % kNS), kBoth);
          }
        }
      }
      // every MMA issued is complete in both CTAs before their epilogues
      // read O and before the tensor memory is released
      for (int q = 0; q < NQ; ++q) ptx::mma_commit2_mc(PB(kPbODone + q), kBoth);
      int drained = 0;
      wait_bar_pair(PB(kPbODone), 0, lim, &drained, p.status, peer_abort);
    } else if (lane == 0) {
      // CTA 1: relay this CTA's TMA completions (and its query extension
      // rows) to CTA 0's MMA thread
      bool ok = wait(PB(kPbQ), 0) && wait(PB(kPbQx), 0);
      if (ok) ptx::mbar_arrive_cluster(LB(kPbQPeer));
      for (int j = n_ct; j < n_t && ok; ++j) {
        if (j == n_ct) {
          if (!(ok = wait(PB(kPbQ), 1))) break;
          ptx::mbar_arrive_cluster(LB(kPbQPeer));
        }
        const int s = j % kNS;
        if (!(ok = wait(PB(kPbFullTma + s), tma_use(j) & 1))) break;
        ptx::mbar_arrive_cluster(LB(kPbTmaPeer + s));
      }
    }
    __syncwarp();
  } else {
    // ============================== TMA ==============================
    if (lane == 0) {
      const uint32_t s_base = ptx::smem_u32(smem);
      auto q_row = [&](int q) { return min(row_base(q), p.n_q - 1); };
      ptx::mbar_expect_tx(PB(kPbQ), NQ * (PRECISE ? 2 : 1) * 2 * kHalf);
      for (int q = 0; q < NQ; ++q) {
        for (int h = 0; h < 2; ++h) {
          ptx::tma_load_3d(s_base + C::kQ + q * C::kTileQ + h * kHalf, &tm_q, 64 * h, q_row(q), bh,
                           PB(kPbQ));
          if (PRECISE)
            ptx::tma_load_3d(s_base + C::kQ + (NQ + q) * C::kTileQ + h * kHalf, &tm_qlo, 64 * h,
                             q_row(q), bh, PB(kPbQ));
        }
      }
      int last = -1;
      bool q_orig_issued = false;
      for (int j = n_ct; j < n_t; ++j) {
        if (*abort) break;
        const int s = j % kNS;
        if (j == n_ct) {
          if (!wait(PB(kPbQFree), 0)) break;
          ptx::mbar_expect_tx(PB(kPbQ), NQ * 2 * kHalf);
          for (int q = 0; q < NQ; ++q)
            for (int h = 0; h < 2; ++h)
              ptx::tma_load_3d(s_base + C::kQ + q * C::kTileQ + h * kHalf, &tm_qo, 64 * h, q_row(q),
                               bh, PB(kPbQ));
          q_orig_issued = true;
        }
        // the V half's barrier: its commit follows the K half's
        if (j >= kNS && !wait(PB(kPbEmptyV + s), ((j / kNS) - 1) & 1)) break;
        const int key0 = (cb + j - n_ct) * kBlockN;
        // this CTA's 64 keys; a half that starts past the last key is loaded
        // from the last key instead (no box lies wholly outside the tensor):
        // its columns are past the valid ones and masked in the softmax
        const int krow = min(key0 + 64 * (int)rank, p.n_r - 1);
        const uint32_t st = s_base + C::kStages + s * C::kStageBytes;
        ptx::mbar_expect_tx(PB(kPbFullTma + s), C::kKTile + (mass_only ? 0 : C::kVTile));
        for (int h = 0; h < 2; ++h)
          ptx::tma_load_3d(st + h * C::kKSub, &tm_k64, 64 * h, krow, bh, PB(kPbFullTma + s));
        if (!mass_only)
          ptx::tma_load_3d(st + C::kV, &tm_v, 64 * (int)rank, key0, bh, PB(kPbFullTma + s));
        last = j;
      }
      if (*abort) {
        int ignore = 0;
        wait_bar_pair(PB(kPbQ), q_orig_issued ? 1 : 0, lim, &ignore, p.status, peer_abort);
        if (last >= 0)
          wait_bar_pair(PB(kPbFullTma + last % kNS), tma_use(last) & 1, lim, &ignore, p.status,
                        peer_abort);
      }
    }
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  // both CTAs done with the pair's MMAs, shared memory and barriers
  ptx::cluster_sync();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc2(tmem, C::kTCols);
  }
#undef PB
#undef LB
}

// One launch of the pair kernel (the dispatcher launches the merge of a
// key-range split); select as in AttnParams.
template <int BITS, int GROUP, int NQ, bool PRECISE>
kvq_status launch_pair_t(const AttnLaunch& a, cudaStream_t stream, int select) {
  using C = PairCfg<NQ, PRECISE>;
  constexpr int D = 128;
  static std::atomic<uint64_t> limit_set{0};
  auto kern = attn_pair_kernel<BITS, GROUP, NQ, PRECISE>;
  if (ensure_smem_limit(kern, C::kAlloc, limit_set) != cudaSuccess) return KVQ_ERR_CUDA;
  CUtensorMap mq, mqlo, mqo, mk, mv;
  if (!make_map(&mq, a.q_rot, D, a.n_q, a.bh, false)) return KVQ_ERR_CUDA;
  if (!make_map(&mqlo, a.q_rot_lo, D, a.n_q, a.bh, false)) return KVQ_ERR_CUDA;
  if (!make_map(&mqo, a.q_orig, D, a.n_q, a.bh, true)) return KVQ_ERR_CUDA;
  if (a.n_r > 0) {
    if (!make_map(&mk, a.k_cur, D, a.n_r, a.bh, true, 64)) return KVQ_ERR_CUDA;
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
  p.status = a.status;
  p.bounds_site = a.bounds_site;
  p.select = select;
  p.select_scale = a.scale * (1.0f / 4096.0f);
  p.qn2 = a.qn2;
  p.kn2 = a.kn2;
  const unsigned pairs = (unsigned)((a.n_q + 2 * kBlockM * NQ - 1) / (2 * kBlockM * NQ));
  const dim3 grid(2 * pairs, a.bh, split ? a.splits : 1);
  kern<<<grid, C::kThreads, C::kAlloc, stream>>>(mq, mqlo, mqo, mk, mv, p);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace

}  // namespace kvq
