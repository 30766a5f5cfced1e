// extern "C" entry points of libkvq: argument validation, the sliding-window
// ring bookkeeping, workspace carving and kernel dispatch.  Every check here
// runs on the host before anything is launched.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "kvq_internal.h"

namespace {

std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---- launch timing (kvq_profile_begin / kvq_profile_end) ----
constexpr int kKinds = 3;
constexpr int kMaxPairs = 16384;
struct Profiler {
  bool on = false;
  std::vector<cudaEvent_t> pool[kKinds];  // 2 events per launch
  int used[kKinds] = {0, 0, 0};
};
Profiler g_prof;
std::atomic<long long> g_kernel_launches{0};

struct ProfScope {
  int kind;
  cudaStream_t s;
  bool active;
  ProfScope(int k, cudaStream_t st) : kind(k), s(st), active(false) {
    if (!g_prof.on || g_prof.used[k] >= kMaxPairs) return;
    auto& pool = g_prof.pool[k];
    const size_t need = 2 * (size_t)(g_prof.used[k] + 1);
    while (pool.size() < need) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return;
      pool.push_back(e);
    }
    if (cudaEventRecord(pool[2 * g_prof.used[k]], s) == cudaSuccess) active = true;
  }
  ~ProfScope() {
    if (!active) return;
    if (cudaEventRecord(g_prof.pool[kind][2 * g_prof.used[kind] + 1], s) == cudaSuccess)
      ++g_prof.used[kind];
  }
};

kvq_status check_geometry(const kvq_cache* c, kvq::Geometry* g) {
  if (c == nullptr) return KVQ_ERR_INVALID_ARG;
  if (c->batch < 1 || c->heads < 1 || c->chunk_tokens < 1 || c->n_chunks < 1)
    return KVQ_ERR_INVALID_ARG;
  if (c->head_dim != 64 && c->head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if (c->bits != 2 && c->bits != 4) return KVQ_ERR_UNSUPPORTED;
  if (c->group != 32 && c->group != 64) return KVQ_ERR_UNSUPPORTED;
  if (c->group > c->head_dim) return KVQ_ERR_UNSUPPORTED;
  const long long bh = (long long)c->batch * c->heads;
  const long long cap = (long long)c->chunk_tokens * c->n_chunks;
  if (bh > (1 << 16) || cap > (1LL << 30) || bh * cap > (1LL << 40)) return KVQ_ERR_INVALID_ARG;
  if (c->len < 0 || c->len > cap || c->head_slot < 0 || c->head_slot >= c->n_chunks)
    return KVQ_ERR_INVALID_ARG;
  if (c->key_mode != KVQ_KEYS_PER_TOKEN && c->key_mode != KVQ_KEYS_PER_CHANNEL)
    return KVQ_ERR_INVALID_ARG;
  g->bh = (int)bh;
  g->d = c->head_dim;
  g->bits = c->bits;
  g->group = c->group;
  g->g = c->head_dim / c->group;
  g->cap = (int)cap;
  g->code_bytes = c->head_dim * c->bits / 8;
  g->key_mode = c->key_mode;
  g->bpc = (c->chunk_tokens + KVQ_KEY_BLOCK - 1) / KVQ_KEY_BLOCK;
  return KVQ_OK;
}

// bytes of k_sz and v_sz
void meta_bytes(const kvq::Geometry& g, int n_chunks, size_t* k, size_t* v) {
  *v = (size_t)g.bh * g.cap * g.g * 4;
  *k = g.key_mode == KVQ_KEYS_PER_CHANNEL ? (size_t)g.bh * n_chunks * g.bpc * g.d * 4 : *v;
}

kvq_status check_cache_buffers(const kvq_cache* c) {
  if (!c->k_codes || !c->v_codes || !c->k_sz || !c->v_sz) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(c->k_codes) || !aligned16(c->v_codes) || !aligned16(c->k_sz) ||
      !aligned16(c->v_sz))
    return KVQ_ERR_ALIGNMENT;
  return KVQ_OK;
}

struct Workspace {
  uint16_t* q_hi;  // rotated queries, FP16
  uint16_t* q_lo;  // FP16 remainder of the rotated queries
  uint16_t* v;     // rotated current-chunk values, FP16
  float* o_part;   // key-range split: partial O, fp32 (splits > 1)
  float* st_part;  // key-range split: base and sums per row (splits > 1)
  float* kch_c;    // per-channel keys: correction per row and cached tile
  float* qn2;      // per head: max ||q'||^2 (the kernel choice of kModeAuto)
  float* kn2;      // per head: max key-norm bound (the same)
  size_t bytes;
};

// the largest number of cached tiles a window of this cache can have
int max_cached_tiles(const kvq::Geometry& g, int n_chunks, int chunk) {
  return kvq::cached_tiles(g.key_mode, n_chunks * chunk, chunk, g.bpc);
}

// kch_tiles: cached tiles the per-(row, tile) table of per-channel keys holds
// (0 without them)
Workspace carve(void* base, const kvq::Geometry& g, int n_q, int n_r, int splits, int kch_tiles) {
  Workspace w;
  const size_t qb = round_up((size_t)g.bh * n_q * g.d * 2, 256);
  const size_t rb = round_up((size_t)g.bh * n_r * g.d * 2, 256);
  const size_t ob = splits > 1 ? round_up((size_t)splits * g.bh * n_q * g.d * 4, 256) : 0;
  const size_t sb = splits > 1 ? round_up((size_t)splits * g.bh * n_q * 3 * 4, 256) : 0;
  const size_t cb = round_up((size_t)kch_tiles * g.bh * n_q * 4, 256);
  const size_t nb = round_up((size_t)g.bh * 4, 256);
  uint8_t* p = static_cast<uint8_t*>(base);
  w.q_hi = reinterpret_cast<uint16_t*>(p);
  w.q_lo = reinterpret_cast<uint16_t*>(p + qb);
  w.v = reinterpret_cast<uint16_t*>(p + 2 * qb);
  w.o_part = reinterpret_cast<float*>(p + 2 * qb + rb);
  w.st_part = reinterpret_cast<float*>(p + 2 * qb + rb + ob);
  w.kch_c = reinterpret_cast<float*>(p + 2 * qb + rb + ob + sb);
  w.qn2 = reinterpret_cast<float*>(p + 2 * qb + rb + ob + sb + cb);
  w.kn2 = reinterpret_cast<float*>(p + 2 * qb + rb + ob + sb + cb + nb);
  w.bytes = 2 * qb + rb + ob + sb + cb + 2 * nb;
  return w;
}

int device_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

// workspace for any kernel shape (one-CTA or SM-pair kernel, one or two
// query tiles per CTA), with room for the split the current device takes on
// a full window (n_s = the cache's capacity); a shorter window whose best
// split needs more room takes the best split that fits
size_t workspace_bytes_any(const kvq::Geometry& g, int n_q, int n_ct, int n_r) {
  const int sms = device_sm_count();
  const int kch = g.key_mode == KVQ_KEYS_PER_CHANNEL ? n_ct : 0;
  size_t best = 0;
  for (int mode = kvq::kModeOneCta; mode <= kvq::kModePair; ++mode) {
    for (int one_tile = 0; one_tile < 2; ++one_tile) {
      const kvq::AttnShape sh =
          kvq::attention_shape(g.bh, n_q, n_ct, n_r, g.d, mode, one_tile != 0, sms, 64);
      const size_t b = carve(nullptr, g, n_q, n_r, sh.splits, kch).bytes;
      if (b > best) best = b;
    }
  }
  return best;
}

kvq_status attention_common(const kvq_cache* cache, const uint16_t* q, const uint16_t* k_cur,
                            const uint16_t* v_cur, int32_t n_q, int32_t n_r, float scale,
                            int32_t corr, int32_t flags, void* workspace, size_t workspace_bytes,
                            uint16_t* out, float* p_s, float* p_r, bool mass_only,
                            void* stream) {
  kvq::Geometry g;
  kvq_status st = check_geometry(cache, &g);
  if (st != KVQ_OK) return st;
  if (n_q < 0 || n_r < 0 || n_q > (1 << 30) || n_r > (1 << 30)) return KVQ_ERR_INVALID_ARG;
  if (corr != KVQ_CORR_NONE && corr != KVQ_CORR_TAYLOR && corr != KVQ_CORR_EXACT)
    return KVQ_ERR_INVALID_ARG;
  if ((flags & ~(KVQ_FLAG_PRECISE_QUERY | KVQ_FLAG_NO_KV_SPLIT | KVQ_FLAG_ONE_CTA |
                 KVQ_FLAG_STAGED_WORDS)) != 0)
    return KVQ_ERR_INVALID_ARG;
  const bool precise = (flags & KVQ_FLAG_PRECISE_QUERY) != 0;
  // one query tile per CTA: the precise-query split, or the exact correction
  // computed in the attention kernel (per-channel keys take it from a pre-pass)
  const bool one_tile =
      precise || (corr == KVQ_CORR_EXACT && cache->key_mode != KVQ_KEYS_PER_CHANNEL);
  if (!std::isfinite(scale) || scale <= 0.f) return KVQ_ERR_INVALID_ARG;
  if ((p_s == nullptr) != (p_r == nullptr)) return KVQ_ERR_INVALID_ARG;
  if (mass_only && p_s == nullptr) return KVQ_ERR_INVALID_ARG;
  if (!mass_only && out == nullptr) return KVQ_ERR_INVALID_ARG;
  if (n_q == 0) return KVQ_OK;
  if (cache->len + n_r < 1) return KVQ_ERR_INVALID_ARG;
  if (cache->len > 0) {
    st = check_cache_buffers(cache);
    if (st != KVQ_OK) return st;
  }
  if (q == nullptr || (n_r > 0 && k_cur == nullptr) || (!mass_only && n_r > 0 && v_cur == nullptr))
    return KVQ_ERR_INVALID_ARG;
  if (!aligned16(q) || (k_cur && !aligned16(k_cur)) || (v_cur && !aligned16(v_cur)) ||
      (out && !aligned16(out)) || !aligned16(workspace))
    return KVQ_ERR_ALIGNMENT;
  if (workspace == nullptr) return KVQ_ERR_INVALID_ARG;
  // key-range split when the grid would not fill the device (and the
  // workspace holds the partial results; otherwise one range)
  const int n_ct = kvq::cached_tiles(g.key_mode, cache->len, cache->chunk_tokens, g.bpc);
  // per-channel keys: a table of one number per row and cached tile (the
  // zero-point term and the correction)
  const int kch_tiles = g.key_mode == KVQ_KEYS_PER_CHANNEL ? n_ct : 0;
  // the SM-pair kernel: head_dim 128, per-token keys, Taylor term or none;
  // with the precise-query flag it runs alone, without it each head takes
  // the pair kernel with the precise split or the one-CTA kernel without,
  // as the GPU finds from the head's norms (kvq::kPreciseSelect)
  const bool pair_ok = g.d == 128 && g.key_mode == KVQ_KEYS_PER_TOKEN && corr != KVQ_CORR_EXACT &&
                       (flags & KVQ_FLAG_ONE_CTA) == 0;
  const int mode = !pair_ok ? kvq::kModeOneCta : precise ? kvq::kModePair : kvq::kModeAuto;
  int max_splits = 1;
  if ((flags & KVQ_FLAG_NO_KV_SPLIT) == 0) {
    max_splits = 64;
    while (max_splits > 1 &&
           carve(nullptr, g, n_q, n_r, max_splits, kch_tiles).bytes > workspace_bytes)
      --max_splits;
  }
  const kvq::AttnShape shape = kvq::attention_shape(g.bh, n_q, n_ct, n_r, g.d, mode, one_tile,
                                                    device_sm_count(), max_splits);
  const int splits = shape.splits, per = shape.tiles_per_split;
  const Workspace ws = carve(workspace, g, n_q, n_r, splits, kch_tiles);
  if (workspace_bytes < ws.bytes) return KVQ_ERR_INVALID_ARG;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = kvq::status_ptr();
  if (status == nullptr) return KVQ_ERR_CUDA;
  // rotate Q (FP16 hi, and lo when the precise split may run) and V_cur
  // (FP16) into the workspace
  kvq::RotateArgs ra{};
  ra.src[0] = q;
  ra.dst[0] = ws.q_hi;
  ra.dst_lo[0] = (precise || mode == kvq::kModeAuto) ? ws.q_lo : nullptr;
  ra.rows[0] = (long long)g.bh * n_q;
  ra.src[1] = v_cur;
  ra.dst[1] = ws.v;
  ra.dst_lo[1] = nullptr;
  ra.rows[1] = mass_only ? 0 : (long long)g.bh * n_r;
  for (int i = 0; i < 4; ++i) ra.sign_bits[i] = cache->sign_bits[i];
  ra.inv_sqrt_d = (float)(1.0 / std::sqrt((double)g.d));
  // FP16 operand limits: every rotated value below 65504; with per-channel
  // keys and the Taylor term the pre-pass squares the query (q'^2 / 64 in
  // FP16): |q'| < 2047
  ra.status = status;
  ra.bounds_site = kvq::bounds_site_ptr();
  ra.range_limit[0] = (g.key_mode == KVQ_KEYS_PER_CHANNEL && corr == KVQ_CORR_TAYLOR) ? 2047.0f
                                                                                     : 65504.0f;
  ra.range_limit[1] = 65504.0f;
  {
    ProfScope prof(1, s);
    // kModeAuto: the per-head norms that choose each head's kernel
    if (mode == kvq::kModeAuto &&
        kvq::launch_select_norms(reinterpret_cast<const uint32_t*>(cache->k_sz), q, g.bh,
                                 cache->len, g.cap, n_q, g.g, g.group, g.bits, ws.kn2, ws.qn2,
                                 s) != cudaSuccess)
      return KVQ_ERR_CUDA;
    if (kvq::launch_rotate(ra, g.d, s) != cudaSuccess) return KVQ_ERR_CUDA;
  }

  kvq::AttnLaunch a{};
  a.k_codes = cache->k_codes;
  a.v_codes = cache->v_codes;
  a.k_sz = reinterpret_cast<const uint32_t*>(cache->k_sz);
  a.v_sz = reinterpret_cast<const uint32_t*>(cache->v_sz);
  a.n_s = cache->len;
  a.cap = g.cap;
  a.q_rot = ws.q_hi;
  a.q_rot_lo = ws.q_lo;
  a.q_orig = q;
  a.k_cur = k_cur;
  a.v_rot = ws.v;
  a.n_q = n_q;
  a.n_r = n_r;
  a.bh = g.bh;
  a.scale = scale;
  a.corr = corr;
  a.precise_query = precise ? 1 : 0;
  a.staged_words = (flags & KVQ_FLAG_STAGED_WORDS) != 0 ? 1 : 0;
  a.mass_only = mass_only ? 1 : 0;
  a.out = out;
  a.p_s = p_s;
  a.p_r = p_r;
  for (int i = 0; i < 4; ++i) a.sign_bits[i] = cache->sign_bits[i];
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.splits = splits;
  a.tiles_per_split = per;
  a.o_part = ws.o_part;
  a.st_part = ws.st_part;
  a.key_mode = g.key_mode;
  a.chunk = cache->chunk_tokens;
  a.bpc = g.bpc;
  a.kblk_per_head = cache->n_chunks * g.bpc;
  a.n_ct = n_ct;
  a.kch_c = kch_tiles > 0 ? ws.kch_c : nullptr;
  a.mode = shape.mode;
  a.qn2 = ws.qn2;
  a.kn2 = ws.kn2;
  ProfScope prof(2, s);
  return kvq::launch_attention(a, g.d, g.bits, g.group, s);
}

}  // namespace

extern "C" {

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported head_dim/bits/group";
    case KVQ_ERR_CAPACITY: return "append refused by the cache window rules";
    case KVQ_ERR_CUDA: return "CUDA call failed";
    case KVQ_ERR_TIMEOUT: return "bounded wait in a kernel ran out";
    case KVQ_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case KVQ_ERR_TOO_LARGE:
      return "problem needs more scratch than kvq_attention_corrected_noalloc's built-in buffer";
    case KVQ_ERR_RANGE:
      return "an operand left the FP16 range of the tensor-core operands (results invalid)";
    case KVQ_ERR_BOUNDS:
      return "checked build: an index left its buffer (see kvq_debug_bounds_site)";
  }
  return "unknown status";
}

int32_t kvq_abi_version(void) { return 2; }

kvq_status kvq_cache_bytes(const kvq_cache* cache, size_t* codes_bytes, size_t* sz_bytes) {
  kvq::Geometry g;
  const kvq_status st = check_geometry(cache, &g);
  if (st != KVQ_OK) return st;
  size_t k = 0, v = 0;
  meta_bytes(g, cache->n_chunks, &k, &v);
  if (codes_bytes) *codes_bytes = (size_t)g.bh * g.cap * g.code_bytes;
  if (sz_bytes) *sz_bytes = k > v ? k : v;
  return KVQ_OK;
}

kvq_status kvq_cache_meta_bytes(const kvq_cache* cache, size_t* k_sz_bytes, size_t* v_sz_bytes) {
  kvq::Geometry g;
  const kvq_status st = check_geometry(cache, &g);
  if (st != KVQ_OK) return st;
  size_t k = 0, v = 0;
  meta_bytes(g, cache->n_chunks, &k, &v);
  if (k_sz_bytes) *k_sz_bytes = k;
  if (v_sz_bytes) *v_sz_bytes = v;
  return KVQ_OK;
}

kvq_status kvq_quantize_append(kvq_cache* cache, const uint16_t* k_new, const uint16_t* v_new,
                               int32_t n_new, void* stream) {
  kvq::Geometry g;
  kvq_status st = check_geometry(cache, &g);
  if (st != KVQ_OK) return st;
  if (n_new < 0) return KVQ_ERR_INVALID_ARG;
  if (n_new > cache->chunk_tokens) return KVQ_ERR_CAPACITY;
  if (n_new == 0) return KVQ_OK;
  if (2LL * g.bh * n_new >= (1LL << 31)) return KVQ_ERR_INVALID_ARG;  // 32-bit row index
  st = check_cache_buffers(cache);
  if (st != KVQ_OK) return st;
  if (k_new == nullptr || v_new == nullptr) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new)) return KVQ_ERR_ALIGNMENT;
  // window rules: fill slots in order, a partial chunk only as the last one,
  // whole chunks only once full
  const int first = cache->head_slot * cache->chunk_tokens;
  int new_len;
  if (cache->len < g.cap) {
    if (cache->len != first) return KVQ_ERR_CAPACITY;
    new_len = cache->len + n_new;
  } else {
    if (n_new != cache->chunk_tokens) return KVQ_ERR_CAPACITY;
    new_len = g.cap;
  }
  kvq::QuantArgs a{};
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_codes = cache->k_codes;
  a.v_codes = cache->v_codes;
  a.k_sz = reinterpret_cast<uint32_t*>(cache->k_sz);
  a.v_sz = reinterpret_cast<uint32_t*>(cache->v_sz);
  a.bh = g.bh;
  a.n_new = n_new;
  a.cap = g.cap;
  a.first = first;
  for (int i = 0; i < 4; ++i) a.sign_bits[i] = cache->sign_bits[i];
  a.inv_sqrt_d = (float)(1.0 / std::sqrt((double)g.d));
  a.v_only = g.key_mode == KVQ_KEYS_PER_CHANNEL ? 1 : 0;
  kvq::row_divisor((uint32_t)n_new, &a.div_mul, &a.div_shift);
  a.kblk_first = cache->head_slot * g.bpc;
  a.kblk_per_head = cache->n_chunks * g.bpc;
  a.status = kvq::status_ptr();
  a.bounds_site = kvq::bounds_site_ptr();
  a.wait_limit_ns = g_wait_limit_ns.load();
  if (a.status == nullptr) return KVQ_ERR_CUDA;
  bool supported = true;
  {
    ProfScope prof(0, static_cast<cudaStream_t>(stream));
    if (kvq::launch_quantize_append_mma(a, g.d, g.bits, g.group,
                                        static_cast<cudaStream_t>(stream),
                                        &supported) != cudaSuccess)
      return KVQ_ERR_CUDA;
    if (!supported) return KVQ_ERR_UNSUPPORTED;
  }
  if (g.key_mode == KVQ_KEYS_PER_CHANNEL) {
    ProfScope prof(0, static_cast<cudaStream_t>(stream));
    if (kvq::launch_quantize_key_channels_mma(a, g.d, g.bits, static_cast<cudaStream_t>(stream),
                                              &supported) != cudaSuccess)
      return KVQ_ERR_CUDA;
    if (!supported) return KVQ_ERR_UNSUPPORTED;
  }
  cache->len = new_len;
  cache->head_slot = (cache->head_slot + 1) % cache->n_chunks;
  return KVQ_OK;
}

size_t kvq_workspace_bytes(const kvq_cache* cache, int32_t n_q, int32_t n_r) {
  kvq::Geometry g;
  if (check_geometry(cache, &g) != KVQ_OK || n_q < 0 || n_r < 0) return 0;
  // the split is sized for a full window (len can only grow up to capacity)
  return workspace_bytes_any(g, n_q, max_cached_tiles(g, cache->n_chunks, cache->chunk_tokens), n_r);
}

kvq_status kvq_attention_corrected(const kvq_cache* cache, const uint16_t* q,
                                   const uint16_t* k_cur, const uint16_t* v_cur, int32_t n_q,
                                   int32_t n_r, float scale, int32_t corr, int32_t flags,
                                   void* workspace, size_t workspace_bytes, uint16_t* out,
                                   float* p_s, float* p_r, void* stream) {
  return attention_common(cache, q, k_cur, v_cur, n_q, n_r, scale, corr, flags, workspace,
                          workspace_bytes, out, p_s, p_r, false, stream);
}

kvq_status kvq_attention_mass(const kvq_cache* cache, const uint16_t* q, const uint16_t* k_cur,
                              int32_t n_q, int32_t n_r, float scale, int32_t corr, int32_t flags,
                              void* workspace, size_t workspace_bytes, float* p_s, float* p_r,
                              void* stream) {
  if (p_s == nullptr || p_r == nullptr) return KVQ_ERR_INVALID_ARG;
  return attention_common(cache, q, k_cur, nullptr, n_q, n_r, scale, corr, flags, workspace,
                          workspace_bytes, nullptr, p_s, p_r, true, stream);
}

kvq_status kvq_rotate(const uint16_t* x, int64_t rows, int32_t d, const uint32_t sign_bits[4],
                      float* out_f32, uint16_t* out_f16, void* stream) {
  if (d != 64 && d != 128) return KVQ_ERR_UNSUPPORTED;
  if (rows < 0 || sign_bits == nullptr) return KVQ_ERR_INVALID_ARG;
  if ((out_f32 == nullptr) == (out_f16 == nullptr)) return KVQ_ERR_INVALID_ARG;
  if (rows == 0) return KVQ_OK;
  if (x == nullptr) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(x) || (out_f32 && !aligned16(out_f32)) || (out_f16 && !aligned16(out_f16)))
    return KVQ_ERR_ALIGNMENT;
  if (out_f32 != nullptr) {
    // the per-token quantizer's rotation (tensor cores), exactly its values
    int* status = kvq::status_ptr();
    if (status == nullptr) return KVQ_ERR_CUDA;
    return kvq::launch_rotate_mma_f32(x, rows, d, sign_bits, out_f32, status,
                                      kvq::bounds_site_ptr(), g_wait_limit_ns.load(),
                                      static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KVQ_OK
               : KVQ_ERR_CUDA;
  }
  kvq::RotateArgs a{};
  a.src[0] = x;
  a.dst[0] = out_f16;
  a.dst_lo[0] = nullptr;
  a.rows[0] = rows;
  a.rows[1] = 0;
  for (int i = 0; i < 4; ++i) a.sign_bits[i] = sign_bits[i];
  a.inv_sqrt_d = (float)(1.0 / std::sqrt((double)d));
  // no FP16 range limits here (range_limit 0); the status word serves the
  // checked build's index checks
  a.status = kvq::status_ptr();
  a.bounds_site = kvq::bounds_site_ptr();
  return kvq::launch_rotate(a, d, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KVQ_OK
                                                                                    : KVQ_ERR_CUDA;
}

kvq_status kvq_last_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVQ_ERR_CUDA;
  int st = 0;
  if (kvq::read_and_clear_attention_status(&st) != KVQ_OK) return KVQ_ERR_CUDA;
  return static_cast<kvq_status>(st);
}

kvq_status kvq_debug_bounds_site(int32_t* line, void* stream) {
  if (line == nullptr) return KVQ_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVQ_ERR_CUDA;
  int v = 0;
  if (kvq::read_and_clear_bounds_site(&v) != KVQ_OK) return KVQ_ERR_CUDA;
  *line = v;
  return KVQ_OK;
}

int32_t kvq_debug_bounds_build(void) {
#ifdef KVQ_DEBUG_BOUNDS
  return 1;
#else
  return 0;
#endif
}

kvq_status kvq_set_wait_limit_ns(uint64_t limit_ns) {
  if (limit_ns == 0) return KVQ_ERR_INVALID_ARG;
  g_wait_limit_ns.store(limit_ns);
  return KVQ_OK;
}

kvq_status kvq_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > 10000000000ull) return KVQ_ERR_INVALID_ARG;
  int* status = kvq::status_ptr();
  if (status == nullptr) return KVQ_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the attention kernels' wait and the tensor-core quantizer's, one after the other
  if (kvq::launch_wait_selftest(limit_ns, s) != cudaSuccess) return KVQ_ERR_CUDA;
  return kvq::launch_quant_wait_selftest(limit_ns, status, s) == cudaSuccess ? KVQ_OK
                                                                             : KVQ_ERR_CUDA;
}

kvq_status kvq_profile_begin(void) {
  for (int k = 0; k < kKinds; ++k) g_prof.used[k] = 0;
  g_kernel_launches.store(0);
  g_prof.on = true;
  return KVQ_OK;
}

int64_t kvq_profile_kernel_launches(void) { return g_kernel_launches.load(); }

kvq_status kvq_profile_end(double ms_total[3], int32_t launches[3]) {
  g_prof.on = false;
  kvq_status st = KVQ_OK;
  for (int k = 0; k < kKinds; ++k) {
    double tot = 0.0;
    for (int i = 0; i < g_prof.used[k]; ++i) {
      float ms = 0.f;
      if (cudaEventSynchronize(g_prof.pool[k][2 * i + 1]) != cudaSuccess ||
          cudaEventElapsedTime(&ms, g_prof.pool[k][2 * i], g_prof.pool[k][2 * i + 1]) !=
              cudaSuccess) {
        st = KVQ_ERR_CUDA;
        continue;
      }
      tot += ms;
    }
    if (ms_total) ms_total[k] = tot;
    if (launches) launches[k] = g_prof.used[k];
    g_prof.used[k] = 0;
  }
  return st;
}

}  // extern "C"

// ---- device addresses of the library's __device__ variables -----------------

namespace {

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// unique id of the calling thread's current context (false when there is
// none yet or the driver does not offer the query)
bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  if (get_current == nullptr || get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

}  // namespace

namespace kvq {

void note_launch() {
  if (g_prof.on) g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
}

cudaError_t device_symbol_address(const void* symbol, SymbolSlot& slot, void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned long long id = 0;
  const bool have_id = current_context_id(&id);
  std::lock_guard<std::mutex> lock(slot.mu);
  if (have_id && slot.ptr[dev] != nullptr && slot.ctx_id[dev] == id) {
    *out = slot.ptr[dev];
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, symbol);
  if (e != cudaSuccess) return e;
  if (p == nullptr) return cudaErrorInvalidSymbol;
  // the lookup itself may have created the context: take its id afterwards
  // (without an id the address is not kept, and every call looks it up)
  unsigned long long id_after = 0;
  if (current_context_id(&id_after)) {
    slot.ctx_id[dev] = id_after;
    slot.ptr[dev] = p;
  } else {
    slot.ptr[dev] = nullptr;
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace kvq

// ---- attention without a workspace argument ---------------------------------
// Scratch of kvq_attention_corrected_noalloc: one fixed device buffer, present
// on every device that loads the library until the process exits.  In host
// code this name is only a host-side stand-in; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

namespace {

kvq::SymbolSlot g_noalloc_slot;

// Device address of the scratch buffer in the current device's current
// context (looked up with that device current, once per device and context).
kvq_status noalloc_scratch(void** ptr) {
  return kvq::device_symbol_address(&g_noalloc_scratch, g_noalloc_slot, ptr) == cudaSuccess
             ? KVQ_OK
             : KVQ_ERR_CUDA;
}

}  // namespace

extern "C" kvq_status kvq_attention_corrected_noalloc(const kvq_cache* cache, const uint16_t* q,
                                                      const uint16_t* k_cur, const uint16_t* v_cur,
                                                      int32_t n_q, int32_t n_r, float scale,
                                                      int32_t corr, int32_t flags, uint16_t* out,
                                                      float* p_s, float* p_r, void* stream) {
  kvq::Geometry g;
  const kvq_status st = check_geometry(cache, &g);
  if (st != KVQ_OK) return st;
  if (n_q < 0 || n_r < 0) return KVQ_ERR_INVALID_ARG;
  const int kch_tiles = g.key_mode == KVQ_KEYS_PER_CHANNEL
                            ? kvq::cached_tiles(g.key_mode, cache->len, cache->chunk_tokens, g.bpc)
                            : 0;
  if (carve(nullptr, g, n_q, n_r, 1, kch_tiles).bytes > (size_t)KVQ_NOALLOC_SCRATCH_BYTES)
    return KVQ_ERR_TOO_LARGE;
  void* scratch = nullptr;
  const kvq_status sst = noalloc_scratch(&scratch);
  if (sst != KVQ_OK) return sst;
  return attention_common(cache, q, k_cur, v_cur, n_q, n_r, scale, corr, flags, scratch,
                          (size_t)KVQ_NOALLOC_SCRATCH_BYTES, out, p_s, p_r, false, stream);
}
