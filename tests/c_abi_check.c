/* A plain C11 caller of libkvq: includes the public header (no C++), links
 * the library and calls the host-only entry points (no GPU needed): ABI
 * version, status strings, cache and metadata sizes in both key modes, and
 * argument errors returned before any launch.  Prints "ok" and exits 0. */
#include <stdio.h>
#include <string.h>

#include "kvq.h"

#define CHECK(c)                                               \
  do {                                                         \
    if (!(c)) {                                                \
      printf("check failed: %s (line %d)\n", #c, __LINE__);   \
      return 1;                                                \
    }                                                          \
  } while (0)

int main(void) {
  kvq_cache c;
  size_t codes = 0, sz = 0, k = 0, v = 0;
  CHECK(kvq_abi_version() == 2);
  CHECK(strcmp(kvq_status_string(KVQ_OK), "ok") == 0);
  memset(&c, 0, sizeof c);
  c.batch = 1;
  c.heads = 24;
  c.head_dim = 128;
  c.bits = 2;
  c.group = 32;
  c.chunk_tokens = 4680;
  c.n_chunks = 4;
  CHECK(kvq_cache_bytes(&c, &codes, &sz) == KVQ_OK);
  CHECK(codes == (size_t)24 * 18720 * 32);
  CHECK(sz == (size_t)24 * 18720 * 4 * 4);
  c.key_mode = KVQ_KEYS_PER_CHANNEL;
  CHECK(kvq_cache_meta_bytes(&c, &k, &v) == KVQ_OK);
  CHECK(k == (size_t)24 * 4 * 37 * 128 * 4 && v == sz);
  c.key_mode = 5;
  CHECK(kvq_cache_bytes(&c, &codes, &sz) == KVQ_ERR_INVALID_ARG);
  c.key_mode = KVQ_KEYS_PER_TOKEN;
  c.head_dim = 96;
  CHECK(kvq_cache_bytes(&c, &codes, &sz) == KVQ_ERR_UNSUPPORTED);
  c.head_dim = 128;
  /* refused on the host before anything touches device memory */
  CHECK(kvq_quantize_append(NULL, NULL, NULL, 1, NULL) == KVQ_ERR_INVALID_ARG);
  CHECK(kvq_attention_corrected(&c, NULL, NULL, NULL, 10, 10, 0.1f, 9, 0, NULL, 0, NULL, NULL,
                                NULL, NULL) == KVQ_ERR_INVALID_ARG);
  printf("ok\n");
  return 0;
}
