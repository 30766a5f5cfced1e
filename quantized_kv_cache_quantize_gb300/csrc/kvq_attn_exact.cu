// Attention kernel instances for the exact correction (sum_c log(sinh a_c / a_c) per cached score, per-token keys).
#include "kvq_attn_kernel.cuh"

namespace kvq {

namespace {

template <int D, int BITS, int GROUP>
kvq_status launch_mode_exact(const AttnLaunch& a, cudaStream_t stream) {
  if (a.precise_query) return launch_t<D, BITS, GROUP, 1, true, true, false>(a, stream);
  return launch_t<D, BITS, GROUP, 1, false, true, false>(a, stream);
}

}  // namespace

kvq_status launch_attention_exact(const AttnLaunch& a, int d, int bits, int group, cudaStream_t stream) {
#define KVQ_A(D_, B_, G_) \
  if (d == D_ && bits == B_ && group == G_) return launch_mode_exact<D_, B_, G_>(a, stream);
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
