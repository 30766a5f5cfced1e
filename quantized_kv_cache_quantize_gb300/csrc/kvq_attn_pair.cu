// Instances and dispatch of the SM-pair attention kernel (kvq_attn_pair.cuh)
// as the library runs it: head_dim 128, per-token keys, no correction or the
// Taylor term, the precise-query split, two query tiles per CTA.  (Measured
// on one GB300: with one query tile per CTA the pair kernel took 1.9x the
// time of two; without the precise split the one-CTA kernel is faster, so
// the pair kernel serves the precise split only.)
#include "kvq_attn_pair.cuh"

namespace kvq {

kvq_status launch_attention_pair(const AttnLaunch& a, int bits, int group, int select,
                                 cudaStream_t stream) {
  if (bits == 2 && group == 32) return launch_pair_t<2, 32, 2, true>(a, stream, select);
  if (bits == 2 && group == 64) return launch_pair_t<2, 64, 2, true>(a, stream, select);
  if (bits == 4 && group == 32) return launch_pair_t<4, 32, 2, true>(a, stream, select);
  if (bits == 4 && group == 64) return launch_pair_t<4, 64, 2, true>(a, stream, select);
  return KVQ_ERR_UNSUPPORTED;
}

}  // namespace kvq
