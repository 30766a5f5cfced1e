// Attention kernel instances for per-channel keys (every correction mode,
// through the per-(row, tile) pre-pass), and the pre-pass kernels.
#include "kvq_attn_kernel.cuh"

namespace kvq {

namespace {

// ---- per-channel keys: zero points and correction per query row and tile ----
//
// A per-channel key tile holds (code - o) * D_c (o the key code offset); what
// its scores still need is the zero-point term scale * sum_c q'_c (o - z_c)
// D_c minus the correction, and with
// per-channel steps both depend on the key only through its block: the
// correction is b = sum_c a_c^2 / 6 (Taylor; = scale^2 / 24 sum_c q'_c^2 D_c^2)
// or sum_c log(sinh a_c / a_c) (exact), a_c = scale/2 |q'_c| D_c, 0 without.
// The table log2(e) (zero-point term - b) [row][tile] is a small GEMM over the
// channels: a CTA covers kKchRows query rows x kKchCols cached tiles of one
// head, each thread a 4 x 4 block of it, with the channels staged through
// shared memory 32 at a time (fp32, with the rotated query the tensor cores
// read: FP16, plus its remainder with the precise-query split).
struct KchArgs {
  const uint16_t* q_hi;   // rotated query, FP16 [bh][n_q][D]
  const uint16_t* q_lo;   // its FP16 remainder, or null
  const uint32_t* k_sz;   // per-channel (step, zero) words [bh][kblk_per_head][D]
  float* out;             // [bh][n_ct][n_q]
  int n_q, n_ct, bpc, kblk_per_head;
  float scale;
  int corr;
  int* status;            // device status word (the tensor-core form's bounded waits)
  float code_offset;      // key tiles hold (code - code_offset) * D_c
  unsigned long long wait_limit_ns;   // limit of every bounded wait
};
constexpr int kKchRows = 64;
constexpr int kKchCols = 32;
constexpr int kKchThreads = (kKchRows / 4) * (kKchCols / 4);   // 128
constexpr int kKchPad = 4;   // shared-memory row padding (floats)

template <int D>
__global__ void __launch_bounds__(kKchThreads) kch_bias_kernel(const KchArgs a) {
  __shared__ __align__(16) float qs[32][kKchRows + kKchPad];   // q'_c of the rows
  __shared__ __align__(16) float wz[32][kKchCols + kKchPad];   // (o - z_c) D_c of the tiles
  __shared__ __align__(16) float wd[32][kKchCols + kKchPad];   // scale/2 D_c of the tiles
  const int tid = threadIdx.x;
  const int ty = tid / (kKchCols / 4), tx = tid % (kKchCols / 4);
  const int row0 = blockIdx.x * kKchRows, t0 = blockIdx.y * kKchCols, bh = blockIdx.z;
  const bool exact = a.corr == KVQ_CORR_EXACT, taylor = a.corr == KVQ_CORR_TAYLOR;
  float az[4][4], ab[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int k = 0; k < 4; ++k) az[i][k] = ab[i][k] = 0.f;
  for (int c0 = 0; c0 < D; c0 += 32) {
    // rows: 64 x 32 channels, 8 channels (16 bytes) per load
    for (int i = tid; i < kKchRows * 4; i += kKchThreads) {
      const int rr = i >> 2, part = i & 3, row = row0 + rr;
      float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (row < a.n_q) {
        const size_t off = ((size_t)bh * a.n_q + row) * D + c0 + 8 * part;
        const uint4 h = __ldg(reinterpret_cast<const uint4*>(a.q_hi + off));
        const uint4 l = a.q_lo ? __ldg(reinterpret_cast<const uint4*>(a.q_lo + off)) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t hw[4] = {h.x, h.y, h.z, h.w}, lw[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          v[2 * k] = h_lo(hw[k]) + h_lo(lw[k]);
          v[2 * k + 1] = h_hi(hw[k]) + h_hi(lw[k]);
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) qs[8 * part + e][rr] = v[e];
    }
    // tiles: 32 x 32 channels of (step, zero) words
    for (int i = tid; i < kKchCols * 4; i += kKchThreads) {
      const int tt = i >> 2, part = i & 3, t = t0 + tt;
      uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      if (t < a.n_ct) {
        const int slot = t / a.bpc;
        const uint4* src = reinterpret_cast<const uint4*>(
            a.k_sz + ((size_t)bh * a.kblk_per_head + slot * a.bpc + (t - slot * a.bpc)) * D + c0 + 8 * part);
        const uint4 x0 = __ldg(src), x1 = __ldg(src + 1);
        w[0] = x0.x; w[1] = x0.y; w[2] = x0.z; w[3] = x0.w;
        w[4] = x1.x; w[5] = x1.y; w[6] = x1.z; w[7] = x1.w;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        wz[8 * part + e][tt] = (a.code_offset - bf16_hi(w[e])) * bf16_lo(w[e]);   // exact: integer, 8-bit step
        wd[8 * part + e][tt] = 0.5f * a.scale * bf16_lo(w[e]);
      }
    }
    __syncthreads();
#pragma unroll 4
    for (int c = 0; c < 32; ++c) {
      const float4 q4 = *reinterpret_cast<const float4*>(&qs[c][4 * ty]);
      const float4 z4 = *reinterpret_cast<const float4*>(&wz[c][4 * tx]);
      const float4 d4 = *reinterpret_cast<const float4*>(&wd[c][4 * tx]);
      const float qv[4] = {q4.x, q4.y, q4.z, q4.w};
      const float zv[4] = {z4.x, z4.y, z4.z, z4.w};
      const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          az[i][k] = fmaf(qv[i], zv[k], az[i][k]);
          if (taylor) {
            const float x = qv[i] * dv[k];
            ab[i][k] = fmaf(x, x, ab[i][k]);
          } else if (exact) {
            ab[i][k] += log_sinhc(fabsf(qv[i]) * dv[k]);
          }
        }
    }
    __syncthreads();
  }
  const float bscale = taylor ? 1.0f / 6.0f : 1.0f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int t = t0 + 4 * tx + k;
    if (t >= a.n_ct) continue;
    float* dst = a.out + ((size_t)bh * a.n_ct + t) * a.n_q;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = row0 + 4 * ty + i;
      if (row < a.n_q) dst[row] = kLog2e * (a.scale * az[i][k] - bscale * ab[i][k]);
    }
  }
}

// The same table on the tensor cores (no correction, or the Taylor term): per
// (query row, cached tile) it is a dot product over a K of parts of D
// channels each,
//   part 0: q_hi . v_hi     part 1: q_hi . v_lo     part 2: q_lo . v_hi (precise)
//   part 3: (q'^2 2^-6) . (u 2^6)                   (Taylor)
// with v = scale log2(e) (o - z_c) D_c split into FP16 high and low parts (the
// products exact in the fp32 accumulator) and u = -log2(e) (scale/2)^2 D_c^2
// / 6.  One CTA: 128 query rows x up to kKgN cached tiles (MMA N), K
// streamed through shared memory 64 channels at a time.
constexpr int kKgN = 128;
constexpr int kKgThreads = 256;   // two threads per query row

template <int D>
__global__ void __launch_bounds__(kKgThreads) kch_gemm_kernel(const KchArgs a) {
  extern __shared__ uint8_t kg_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(kg_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  // two chunk buffers, each A (128 rows x 64 FP16) then B (kKgN rows x 64
  // FP16), 128-byte swizzle: chunk c + 1 is written while the MMAs of chunk
  // c run
  constexpr int kBuf = 128 * 128 + kKgN * 128;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 2 * kBuf);   // [2] chunk MMAs done
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 2);
  volatile int* abort = reinterpret_cast<volatile int*>(bar + 3);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int r = tid & 127, half = tid >> 7;   // row of the tile, half of its channels
  const int row = blockIdx.x * 128 + r;
  const int t0 = blockIdx.y * kKgN, bh = blockIdx.z;
  const int nt = min(kKgN, a.n_ct - t0);
  const int npad = (nt + 15) & ~15;
  const uint32_t bar0 = ptx::smem_u32(bar);
  if (tid == 0) {
    ptx::mbar_init(bar0, 1);
    ptx::mbar_init(bar0 + 8, 1);
    *abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(tslot), kKgN);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tslot;
  const bool taylor = a.corr == KVQ_CORR_TAYLOR;
  const float sl2 = a.scale * kLog2e;
  const float uc = -kLog2e * 0.25f * a.scale * a.scale * (1.0f / 6.0f) * 64.0f;
  const size_t qoff = ((size_t)bh * a.n_q + min(row, a.n_q - 1)) * D;
  const uint32_t idesc = ptx::idesc_f16kind(128, npad, false, false);
  // the chunks: (part, 64-channel block) for the parts this launch needs
  const int np = a.q_lo != nullptr ? 3 : 2;
  const int n_chunks = (np + (taylor ? 1 : 0)) * (D / 64);
  int issued = 0;   // chunks whose MMAs were issued
  for (int ci = 0; ci < n_chunks; ++ci) {
    const int pi = ci / (D / 64), kc = ci - pi * (D / 64);
    const int part = pi < np ? pi : 3;
    const int b = ci & 1;
    uint8_t* ta = sm + b * kBuf;
    uint8_t* tb = ta + 128 * 128;
    // buffer b was last read by the MMAs of chunk ci - 2; if that wait ran
    // out (or another thread's did), no further chunk is written or issued
    bool free_ok = true;
    if (ci >= 2) free_ok = wait_bar(bar0 + 8 * b, ((ci - 2) >> 1) & 1, a.wait_limit_ns, abort, a.status);
    if (!__syncthreads_and(free_ok && !*abort)) break;
    // A: this thread's half of its row's channels [64 kc, 64 kc + 64)
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      const int c8 = 4 * half + c4;
      const int ch = 64 * kc + 8 * c8;
      const uint4 h = __ldg(reinterpret_cast<const uint4*>(a.q_hi + qoff + ch));
      uint4 v = h;
      if (part == 2 || part == 3) {
        const uint4 l = a.q_lo ? __ldg(reinterpret_cast<const uint4*>(a.q_lo + qoff + ch))
                               : make_uint4(0u, 0u, 0u, 0u);
        if (part == 2) {
          v = l;
        } else {
          const uint32_t hw[4] = {h.x, h.y, h.z, h.w}, lw[4] = {l.x, l.y, l.z, l.w};
          uint32_t o[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float x0 = h_lo(hw[k]) + h_lo(lw[k]), x1 = h_hi(hw[k]) + h_hi(lw[k]);
            o[k] = pack_h2(x0 * x0 * (1.0f / 64.0f), x1 * x1 * (1.0f / 64.0f));
          }
          v = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      *reinterpret_cast<uint4*>(ta + sw128(r, c8)) = v;
    }
    // B: rows = cached tiles t0 + n (zero past the last), same channels
    for (int idx = tid; idx < npad * 8; idx += kKgThreads) {
      const int n = idx >> 3, c8 = idx & 7, t = t0 + n;
      uint32_t o[4] = {0u, 0u, 0u, 0u};
      if (n < nt) {
        const int slot = t / a.bpc;
        const uint4* src = reinterpret_cast<const uint4*>(
            a.k_sz + ((size_t)bh * a.kblk_per_head + slot * a.bpc + (t - slot * a.bpc)) * D +
            64 * kc + 8 * c8);
        const uint4 x0 = __ldg(src), x1 = __ldg(src + 1);
        const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float dl = bf16_lo(w[e]);
          if (part == 3) {
            f[e] = uc * dl * dl;
          } else {
            const float vv = sl2 * ((a.code_offset - bf16_hi(w[e])) * dl);
            const float vh = __half2float(__float2half_rn(vv));
            f[e] = part == 1 ? vv - vh : vh;
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) o[k] = pack_h2(f[2 * k], f[2 * k + 1]);
      }
      *reinterpret_cast<uint4*>(tb + sw128(n, c8)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    ptx::fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      ptx::tc_fence_after();
      const uint64_t da = ptx::smem_desc(ptx::smem_u32(ta), 16, 1024, ptx::kLayoutSw128);
      const uint64_t db = ptx::smem_desc(ptx::smem_u32(tb), 16, 1024, ptx::kLayoutSw128);
#pragma unroll
      for (int s4 = 0; s4 < 4; ++s4)
        ptx::mma_f16(tmem, da + (uint64_t)(s4 * 2), db + (uint64_t)(s4 * 2), idesc,
                     (ci > 0 || s4 > 0) ? 1u : 0u);
      ptx::mma_commit(bar0 + 8 * b);
    }
    issued = ci + 1;
  }
  // every MMA issued is complete (the last commit covers the earlier ones)
  // before the tensor memory is read or freed, also after a wait that ran out
  if (issued > 0) {
    const int last = issued - 1;
    int drained = 0;
    wait_bar(bar0 + 8 * (last & 1), (last >> 1) & 1, a.wait_limit_ns, &drained, a.status);
  }
  ptx::tc_fence_after();
  // the tensor-memory loads are warp-collective: every lane of warps 0-3
  // (lanes 0-127: the rows) takes part, only the rows of the chunk store;
  // nothing is read after an aborted chunk loop
  const bool complete = __syncthreads_and(issued == n_chunks && !*abort);
  if (warp < 4 && complete) {
    for (int c = 0; c < npad; c += 32) {
      uint32_t v[32];
      ptx::tmem_ld32(tmem + c + ((uint32_t)(warp * 32) << 16), v);
      if (row < a.n_q) {
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (c + k < nt) a.out[((size_t)bh * a.n_ct + t0 + c + k) * a.n_q + row] = __uint_as_float(v[k]);
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kKgN);
  }
}

// the pre-pass of one launch: the table of zero-point term minus correction
template <int D, int BITS>
kvq_status launch_kch_table(const AttnLaunch& a, cudaStream_t stream) {
  if (a.kch_c == nullptr || a.n_ct <= 0 || a.n_q <= 0) return KVQ_OK;
  KchArgs k;
  k.q_hi = a.q_rot;
  k.q_lo = a.precise_query ? a.q_rot_lo : nullptr;
  k.k_sz = a.k_sz;
  k.out = a.kch_c;
  k.n_q = a.n_q;
  k.n_ct = a.n_ct;
  k.bpc = a.bpc;
  k.kblk_per_head = a.kblk_per_head;
  k.scale = a.scale;
  k.corr = a.corr;
  k.status = a.status;
  k.code_offset = (float)key_code_offset<BITS>();
  k.wait_limit_ns = a.wait_limit_ns;
  if (a.corr == KVQ_CORR_EXACT) {
    // log(sinh a / a) per channel: the CUDA-core form
    const dim3 kg((a.n_q + kKchRows - 1) / kKchRows, (a.n_ct + kKchCols - 1) / kKchCols, a.bh);
    kch_bias_kernel<D><<<kg, kKchThreads, 0, stream>>>(k);
    note_launch();
  } else {
    const dim3 kg((a.n_q + 127) / 128, (a.n_ct + kKgN - 1) / kKgN, a.bh);
    // two 32 KB chunk buffers (at most three CTAs, 3 x 128 tensor-memory
    // columns, share an SM)
    const int smem = 1024 + 2 * (128 * 128 + kKgN * 128) + 64;
    static std::atomic<uint64_t> kg_limit{0};
    if (ensure_smem_limit(kch_gemm_kernel<D>, smem, kg_limit) != cudaSuccess) return KVQ_ERR_CUDA;
    kch_gemm_kernel<D><<<kg, kKgThreads, smem, stream>>>(k);
    note_launch();
  }
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

template <int D, int BITS, int GROUP>
kvq_status launch_mode_kch(const AttnLaunch& a, cudaStream_t stream) {
  const kvq_status st = launch_kch_table<D, BITS>(a, stream);
  if (st != KVQ_OK) return st;
  if (a.precise_query) return launch_t<D, BITS, GROUP, 1, true, false, true>(a, stream);
  return launch_t<D, BITS, GROUP, 2, false, false, true>(a, stream);
}

}  // namespace

kvq_status launch_attention_kch(const AttnLaunch& a, int d, int bits, int group, cudaStream_t stream) {
#define KVQ_A(D_, B_, G_) \
  if (d == D_ && bits == B_ && group == G_) return launch_mode_kch<D_, B_, G_>(a, stream);
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

}  // namespace kvq
