// Index checks of the checked build.
//
// Compiled with -DKVQ_DEBUG_BOUNDS (libkvq_checked.so), KVQ_IN_BOUNDS(i, n,
// status, site) is false when the index i falls outside [0, n): the kernel
// then skips the access, and the first failing check records KVQ_ERR_BOUNDS
// in the device status word and its source line in the site word.  In the
// regular build it is the constant true and costs nothing.
#pragma once

#include "kvq.h"

namespace kvq {

__device__ __forceinline__ bool in_bounds(long long i, long long n, int* status, int* site,
                                          int line) {
#ifdef KVQ_DEBUG_BOUNDS
  if (i >= 0 && i < n) return true;
  if (status != nullptr && atomicCAS(status, 0, (int)KVQ_ERR_BOUNDS) == 0 && site != nullptr)
    atomicExch(site, line);
  return false;
#else
  (void)i; (void)n; (void)status; (void)site; (void)line;
  return true;
#endif
}

}  // namespace kvq

#define KVQ_IN_BOUNDS(i, n, status, site) \
  kvq::in_bounds((long long)(i), (long long)(n), (status), (site), __LINE__)
