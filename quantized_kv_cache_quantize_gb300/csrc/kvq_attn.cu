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
kvq_status launch_mode(const AttnLaunch& a, cudaStream_t stream) {
  if (a.precise_query) return launch_t<D, BITS, GROUP, 1, true, false, false>(a, stream);
  return launch_t<D, BITS, GROUP, 2, false, false, false>(a, stream);
}

SymbolSlot g_status_slot;

}  // namespace

// device address of the status word in the current device's current context
int* status_ptr() {
  void* p = nullptr;
  if (device_symbol_address(&g_attn_status, g_status_slot, &p) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

kvq_status launch_attention(const AttnLaunch& a_in, int d, int bits, int group, cudaStream_t stream) {
  AttnLaunch a = a_in;
  a.status = status_ptr();
  if (a.status == nullptr) return KVQ_ERR_CUDA;
  if (a.key_mode == KVQ_KEYS_PER_CHANNEL) return launch_attention_kch(a, d, bits, group, stream);
  if (a.corr == KVQ_CORR_EXACT) return launch_attention_exact(a, d, bits, group, stream);
#define KVQ_A(D_, B_, G_) \
  if (d == D_ && bits == B_ && group == G_) return launch_mode<D_, B_, G_>(a, stream);
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
