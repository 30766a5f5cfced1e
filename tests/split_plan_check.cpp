// Host-side launch planning of the attention, checked without a GPU.
//
// kvq::attention_split picks how many key-tile ranges each (head, query
// block) is divided into, for one-CTA grids and for SM-pair grids (two CTAs
// per block of twice the rows); kvq::attention_shape plans each kernel mode.  Whatever it picks, the ranges must cover the key
// tiles exactly once with none empty, hold at least two tiles each, stay
// within min(64, max_splits), and leave a grid that already fills whole
// waves of SMs unsplit (splitting it only adds set-up and merge work).
// kvq::cached_tiles must count the 128-token tiles of the window, or with
// per-channel keys the key blocks of every chunk slot.
//
// Mode "sweep": prints "checks N bad M", exits 1 on any violation.
// Mode "tiles": reads lines "key_mode n_s chunk" on stdin and prints the
// tile count of each (compared with the oracle's block partition in Python).
#include <cstdio>
#include <cstring>
#include <random>

#include "../quantized_kv_cache_quantize_gb300/csrc/kvq_internal.h"

static long long bad = 0, checks = 0;

static void fail(const char* what, long long bh, int n_q, int n_ct, int n_r, int rows, int sms,
                 int max_splits, int splits, int per) {
  if (bad < 10)
    std::printf("%s: bh %lld n_q %d n_ct %d n_r %d rows %d sms %d max %d -> splits %d per %d\n",
                what, bh, n_q, n_ct, n_r, rows, sms, max_splits, splits, per);
  ++bad;
}

static void check(long long bh, int n_q, int n_ct, int n_r, int d, int rows, int sms, int max_splits,
                  bool pair = false) {
  int splits = -1, per = -1;
  kvq::attention_split(bh, n_q, n_ct, n_r, d, rows, sms, max_splits, &splits, &per, pair);
  ++checks;
  const int n_t = n_ct + (n_r + 127) / 128;
  if (splits < 1 || per < 1) return fail("non-positive", bh, n_q, n_ct, n_r, rows, sms, max_splits, splits, per);
  if (splits == 1) {
    if (per != (n_t > 0 ? n_t : 1)) fail("unsplit range", bh, n_q, n_ct, n_r, rows, sms, max_splits, splits, per);
    return;
  }
  // every range non-empty, all tiles covered
  if (!((long long)(splits - 1) * per < n_t && n_t <= (long long)splits * per))
    fail("cover", bh, n_q, n_ct, n_r, rows, sms, max_splits, splits, per);
  if (per < 2) fail("range < 2 tiles", bh, n_q, n_ct, n_r, rows, sms, max_splits, splits, per);
  if (splits > 64 || splits > max_splits) fail("too many", bh, n_q, n_ct, n_r, rows, sms, max_splits, splits, per);
  if (n_t < 4) fail("split of < 4 tiles", bh, n_q, n_ct, n_r, rows, sms, max_splits, splits, per);
  const long long ctas = pair ? 2 * bh * ((n_q + 2 * rows - 1) / (2 * rows)) : bh * ((n_q + rows - 1) / rows);
  if (ctas > 0 && ctas % sms == 0) fail("full waves split", bh, n_q, n_ct, n_r, rows, sms, max_splits, splits, per);
}

// the shape chooser: pair shapes only where allowed, one query tile when the
// one-CTA kernel needs it, and the split it reports is the chosen shape's
static void check_shape(long long bh, int n_q, int n_ct, int n_r, int sms, int max_splits) {
  for (int mode = kvq::kModeOneCta; mode <= kvq::kModeAuto; ++mode)
    for (int one_tile = 0; one_tile < 2; ++one_tile) {
      const kvq::AttnShape sh =
          kvq::attention_shape(bh, n_q, n_ct, n_r, 128, mode, one_tile != 0, sms, max_splits);
      ++checks;
      if (sh.mode != mode) fail("mode", bh, n_q, n_ct, n_r, 0, sms, max_splits, sh.splits, sh.tiles_per_split);
      // the one-CTA kernel alone: one query tile when asked; otherwise two
      // (the pair kernel, and the one-CTA kernel beside it in kModeAuto)
      if (sh.nq != (mode == kvq::kModeOneCta && one_tile ? 1 : 2))
        fail("nq", bh, n_q, n_ct, n_r, 0, sms, max_splits, sh.splits, sh.tiles_per_split);
      int sp = 0, per = 0;
      kvq::attention_split(bh, n_q, n_ct, n_r, 128, 128 * sh.nq, sms, max_splits, &sp, &per,
                           mode == kvq::kModePair);
      if (sp != sh.splits || per != sh.tiles_per_split)
        fail("shape split", bh, n_q, n_ct, n_r, 128 * sh.nq, sms, max_splits, sh.splits, sh.tiles_per_split);
    }
}

int main(int argc, char** argv) {
  if (argc > 1 && std::strcmp(argv[1], "tiles") == 0) {
    int mode, n_s, chunk;
    while (std::scanf("%d %d %d", &mode, &n_s, &chunk) == 3) {
      const int bpc = (chunk + kvq::kKeyBlock - 1) / kvq::kKeyBlock;
      std::printf("%d\n", kvq::cached_tiles(mode, n_s, chunk, bpc));
    }
    return 0;
  }
  std::mt19937_64 rng(3);
  const int sms_list[] = {1, 2, 8, 132, 148, 152, 160};
  for (int sms : sms_list)
    for (long long bh : {1LL, 2LL, 3LL, 7LL, 24LL, 32LL, 40LL, 152LL, 1000LL})
      for (int n_q : {1, 60, 127, 128, 129, 256, 300, 4680, 14400})
        for (int n_ct : {0, 1, 2, 3, 4, 5, 33, 147, 148, 391, 676})
          for (int n_r : {0, 1, 128, 300, 4680})
            for (int rows : {128, 256})
              for (int max_splits : {1, 2, 16, 64, 1000})
                for (int pair = 0; pair < 2; ++pair) {
                  check(bh, n_q, n_ct, n_r, 128, rows, sms, max_splits, pair != 0);
                  if (rows == 128 && pair == 0) check_shape(bh, n_q, n_ct, n_r, sms, max_splits);
                }
  for (int i = 0; i < 2000000; ++i) {
    const int sms = 1 + (int)(rng() % 200);
    const long long bh = 1 + (long long)(rng() % 5000);
    const int n_q = 1 + (int)(rng() % 20000);
    const int n_ct = (int)(rng() % 3000);
    const int n_r = (int)(rng() % 20000);
    const int rows = (rng() & 1) ? 128 : 256;
    const int max_splits = 1 + (int)(rng() % 100);
    check(bh, n_q, n_ct, n_r, (rng() & 1) ? 64 : 128, rows, sms, max_splits, (rng() & 1) != 0);
  }
  std::printf("checks %lld bad %lld\n", checks, bad);
  return bad ? 1 : 0;
}
