// Fused Jensen-bias-corrected chunk attention over a low-bit KV window:
// dispatch, the device status word and the bounded-wait self-test.  The
// kernels are in kvq_attn_kernel.cuh; this unit instantiates the per-token
// key modes with the Taylor correction or none, kvq_attn_exact.cu the exact
// correction and kvq_attn_kch.cu the per-channel keys.
#include "kvq_attn_kernel.cuh"

namespace kvq {

namespace {

// first error of a bounded wait in any attention kernel (KVQ_OK if none)
__device__ int g_attn_status;
// checked build: the source line of the first failed index check
__device__ int g_bounds_site;

__global__ void wait_selftest_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t b;
  __shared__ int abort_flag;
  const uint32_t a = ptx::smem_u32(&b);
  if (threadIdx.x == 0) {
    ptx::mbar_init(a, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  // nothing ever arrives on this barrier: the wait must run out and return
  wait_bar(a, 0, limit_ns, &abort_flag, &g_attn_status);
}

template <int D, int BITS, int GROUP>
kvq_status launch_mode(const AttnLaunch& a, cudaStream_t stream, int select) {
  if (a.precise_query) return launch_t<D, BITS, GROUP, 1, true, false, false>(a, stream, select);
  if constexpr (D == 128 && BITS == 2 && GROUP == 32) {
    if (a.staged_words) return launch_t<D, BITS, GROUP, 2, false, false, false, true>(a, stream, select);
  }
  return launch_t<D, BITS, GROUP, 2, false, false, false>(a, stream, select);
}

// the one-CTA kernel for per-token keys, no correction or the Taylor term
kvq_status launch_one_cta(const AttnLaunch& a, int d, int bits, int group, cudaStream_t stream,
                          int select) {
#define KVQ_A(D_, B_, G_) \
  if (d == D_ && bits == B_ && group == G_) return launch_mode<D_, B_, G_>(a, stream, select);
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

// The per-head maxima of kPreciseSelect, one block per (chunk, head) and
// one atomic maximum per block (non-negative floats order like their bit
// patterns; kn2 and qn2 are cleared before the launch).  Blocks
// [0, key_blocks) of grid.x take kSelectTokens cached keys each: thread per
// key, its G (step, zero) words in one load, B^2 = sum_g group *
// (max(|z_g|, 2^bits - 1 - z_g) D_g)^2 >= ||k_hat'||^2.  The other blocks
// take kSelectRows query rows each: 16 lanes per row of 128 BF16 values,
// four rows per lane group in flight, ||q||^2 (= ||q'||^2).
constexpr int kSelectTokens = 2048;
constexpr int kSelectRows = 256;
template <int G>
__global__ void __launch_bounds__(256) select_norms_kernel(const uint32_t* k_sz, const uint16_t* q,
                                                           int n_s, int cap, int n_q,
                                                           int key_blocks, int group, float qmax,
                                                           float* kn2, float* qn2) {
  __shared__ float part[8];
  const int bh = blockIdx.y;
  const bool keys = (int)blockIdx.x < key_blocks;
  float mx = 0.f;
  if (keys) {
    const uint32_t* base = k_sz + (size_t)bh * cap * G;
    const int t0 = blockIdx.x * kSelectTokens;
    const int t1 = min(n_s, t0 + kSelectTokens);
    for (int t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
      uint32_t w[G];
      if (G == 4) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(base + (size_t)t * G));
        w[0] = v.x; w[1 % G] = v.y; w[2 % G] = v.z; w[3 % G] = v.w;
      } else if (G == 2) {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(base + (size_t)t * G));
        w[0] = v.x; w[1 % G] = v.y;
      } else {
        w[0] = __ldg(base + (size_t)t * G);
      }
      float b = 0.f;
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const float m = fmaxf(fabsf(bf16_hi(w[j])), fabsf(qmax - bf16_hi(w[j]))) * bf16_lo(w[j]);
        b = fmaf(m, m, b);
      }
      mx = fmaxf(mx, b * (float)group);
    }
  } else {
    const int r0 = ((int)blockIdx.x - key_blocks) * kSelectRows;
    const int r1 = min(n_q, r0 + kSelectRows);
    const int sub = threadIdx.x & 15;   // 8 channels of the row
    const uint16_t* base = q + (size_t)bh * n_q * 128;
    // every lane runs the same number of iterations (shuffles below); the
    // 16-row steps of four iterations are loaded before any is reduced
    constexpr int kU = 4;
    for (int rb = r0; rb < r1; rb += 16 * kU) {
      uint4 v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int r = rb + 16 * u + (threadIdx.x >> 4);
        v[u] = r < r1 ? __ldg(reinterpret_cast<const uint4*>(base + (size_t)r * 128 + 8 * sub))
                      : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        float n2 = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          n2 = fmaf(bf16_lo(w[i]), bf16_lo(w[i]), n2);
          n2 = fmaf(bf16_hi(w[i]), bf16_hi(w[i]), n2);
        }
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) n2 += __shfl_xor_sync(0xffffffffu, n2, o);
        mx = fmaxf(mx, n2);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) mx = fmaxf(mx, part[i]);
    atomicMax(reinterpret_cast<unsigned int*>((keys ? kn2 : qn2) + bh), __float_as_uint(mx));
  }
}

SymbolSlot g_status_slot;
SymbolSlot g_site_slot;

}  // namespace

// device address of the status word in the current device's current context
int* status_ptr() {
  void* p = nullptr;
  if (device_symbol_address(&g_attn_status, g_status_slot, &p) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

// device address of the checked build's site word (current device and context)
int* bounds_site_ptr() {
  void* p = nullptr;
  if (device_symbol_address(&g_bounds_site, g_site_slot, &p) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

kvq_status read_and_clear_bounds_site(int* line) {
  int zero = 0;
  if (cudaMemcpyFromSymbol(line, g_bounds_site, sizeof(int)) != cudaSuccess) return KVQ_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_bounds_site, &zero, sizeof(int)) != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

cudaError_t launch_select_norms(const uint32_t* k_sz, const uint16_t* q, int bh, int n_s, int cap,
                                int n_q, int g, int group, int bits, float* kn2, float* qn2,
                                cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(kn2, 0, (size_t)bh * sizeof(float), stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(qn2, 0, (size_t)bh * sizeof(float), stream);
  if (e != cudaSuccess) return e;
  const int kblocks = (n_s + kSelectTokens - 1) / kSelectTokens;
  const int qblocks = (n_q + kSelectRows - 1) / kSelectRows;
  if (kblocks + qblocks == 0) return cudaSuccess;
  const dim3 grid((unsigned)(kblocks + qblocks), (unsigned)bh);
  const float qmax = (float)((1 << bits) - 1);
  if (g == 4) {
    select_norms_kernel<4><<<grid, 256, 0, stream>>>(k_sz, q, n_s, cap, n_q, kblocks, group, qmax,
                                                     kn2, qn2);
    note_launch();
  } else if (g == 2) {
    select_norms_kernel<2><<<grid, 256, 0, stream>>>(k_sz, q, n_s, cap, n_q, kblocks, group, qmax,
                                                     kn2, qn2);
    note_launch();
  } else {
    select_norms_kernel<1><<<grid, 256, 0, stream>>>(k_sz, q, n_s, cap, n_q, kblocks, group, qmax,
                                                     kn2, qn2);
    note_launch();
  }
  return cudaGetLastError();
}

kvq_status launch_attention(const AttnLaunch& a_in, int d, int bits, int group, cudaStream_t stream) {
  AttnLaunch a = a_in;
  a.status = status_ptr();
  if (a.status == nullptr) return KVQ_ERR_CUDA;
  a.bounds_site = bounds_site_ptr();
  kvq_status st;
  if (a.mode == kModePair) {
    st = launch_attention_pair(a, bits, group, 0, stream);
  } else if (a.mode == kModeAuto) {
    // every head by one of the two kernels, chosen on the GPU
    AttnLaunch fast = a;
    fast.precise_query = 0;
    st = launch_one_cta(fast, d, bits, group, stream, -1);
    if (st == KVQ_OK) {
      AttnLaunch precise = a;
      precise.precise_query = 1;
      st = launch_attention_pair(precise, bits, group, +1, stream);
    }
  } else if (a.key_mode == KVQ_KEYS_PER_CHANNEL) {
    st = launch_attention_kch(a, d, bits, group, stream);
  } else if (a.corr == KVQ_CORR_EXACT) {
    st = launch_attention_exact(a, d, bits, group, stream);
  } else {
    st = launch_one_cta(a, d, bits, group, stream, 0);
  }
  // the key-range split's partial results, merged once for the whole call
  if (st == KVQ_OK && a.splits > 1) {
    const float inv_sqrt_d = (float)(1.0 / sqrt((double)d));
    st = d == 64 ? launch_merge<64>(a, inv_sqrt_d, stream) : launch_merge<128>(a, inv_sqrt_d, stream);
  }
  return st;
}

kvq_status read_and_clear_attention_status(int* status) {
  int zero = 0;
  if (cudaMemcpyFromSymbol(status, g_attn_status, sizeof(int)) != cudaSuccess) return KVQ_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(int)) != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
  note_launch();
  return cudaGetLastError();
}

}  // namespace kvq
