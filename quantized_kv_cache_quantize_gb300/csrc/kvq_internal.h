// Host-side declarations shared by the translation units of libkvq.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/kvq.h"

namespace kvq {

// Geometry of one cache, validated once per call.
struct Geometry {
  int bh;          // batch * heads
  int d;           // head dim
  int bits;
  int group;
  int g;           // groups per token (d / group)
  int cap;         // tokens per head
  int code_bytes;  // packed bytes per token
  int key_mode;    // KVQ_KEYS_PER_TOKEN / KVQ_KEYS_PER_CHANNEL
  int bpc;         // key blocks per chunk slot (per-channel keys)
};

// Arguments of the quantize-append kernel.
struct QuantArgs {
  const uint16_t* k_new;
  const uint16_t* v_new;
  uint8_t* k_codes;
  uint8_t* v_codes;
  uint32_t* k_sz;  // one 32-bit word (bf16 step | bf16 zero << 16) per group
  uint32_t* v_sz;
  int bh;
  int n_new;
  int cap;
  int first;       // first token written in every head
  uint32_t sign_bits[4];
  float inv_sqrt_d;
  int v_only;      // per-channel key mode: the per-token kernels quantize the V rows only
  // row r of a tensor is token r - n_new * (r / n_new) of (batch, head)
  // r / n_new, the quotient taken as umulhi(r, div_mul) >> div_shift
  // (div_mul = 0: a power of two, r >> div_shift)
  uint32_t div_mul;
  int div_shift;
  // per-channel key mode: k_sz holds kblk_per_head blocks of d words per
  // head; this append's blocks start at block kblk_first
  int kblk_first;
  int kblk_per_head;
  // checked build: where a failed index check is recorded
  int* status;
  int* bounds_site;
  unsigned long long wait_limit_ns;   // bounded waits of the tensor-core quantizer
};

// Arguments of the rotation kernel: up to two row segments in one launch.
// Per segment: FP16 output in dst plus, when dst_lo is set, the FP16
// rounding remainder fp16(x - fp16(x)) in dst_lo.
// With status set, a segment whose range_limit[i] > 0 records KVQ_ERR_RANGE
// there when a rotated value reaches that magnitude (FP16 outputs only).
struct RotateArgs {
  const uint16_t* src[2];
  void* dst[2];
  uint16_t* dst_lo[2];
  long long rows[2];
  uint32_t sign_bits[4];
  float inv_sqrt_d;
  int* status;
  float range_limit[2];
  int* bounds_site;   // checked build: source line of the first failed index check
};

// Raise a kernel's dynamic shared-memory limit once per device (the
// attribute belongs to the current device's context); `done` holds one bit
// per device ordinal below 64.
template <typename Kernel>
cudaError_t ensure_smem_limit(Kernel kern, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t{1} << dev) : 0;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Device address of one of this library's __device__ variables, valid in
// the calling thread's current context.  In host code the variable's name is
// only a host-side stand-in, so the address comes from cudaGetSymbolAddress;
// it is cached per device together with the unique id of the context it was
// looked up in, and looked up again when that context changes (after
// cudaDeviceReset, or with another context made current).  The lookup may
// load the library's device code: the first call on a device, and the first
// after a context change, must come before any stream capture.
constexpr int kMaxDevices = 64;
struct SymbolSlot {
  std::mutex mu;
  unsigned long long ctx_id[kMaxDevices] = {};
  void* ptr[kMaxDevices] = {};
};
cudaError_t device_symbol_address(const void* symbol, SymbolSlot& slot, void** out);

// Multiplier and shift of the quotient r / d for every r < 2^31 and
// 1 <= d < 2^31 (division by an invariant integer, Granlund and Montgomery):
// with l = floor(log2 d), d not a power of two, m = ceil(2^(32+l) / d) fits
// 32 bits and umulhi(r, m) >> l = floor(r / d), because r * (m - 2^(32+l)/d)
// / 2^(32+l) < r / 2^(32+l) < 1/d when r < 2^31 <= 2^(32+l)/d.  A power of
// two is a plain shift (m = 0).
inline void row_divisor(uint32_t d, uint32_t* mul, int* shift) {
  int l = 0;
  while ((2u << l) <= d && l < 31) ++l;   // 2^l <= d < 2^(l+1)
  *shift = l;
  if ((d & (d - 1)) == 0) {
    *mul = 0;
    return;
  }
  const unsigned long long num = 1ull << (32 + l);
  *mul = (uint32_t)((num + d - 1) / d);
}

// per-channel key mode: the K rows of one append, per channel over blocks of
// kKeyBlock tokens
constexpr int kKeyBlock = 128;
cudaError_t launch_rotate(const RotateArgs& a, int d, cudaStream_t stream);
// The per-token quantize-append with the rotation on the tensor cores
// (kvq_quant_mma.cu), and its rotation alone: fp32 x' of `rows` BF16 rows,
// exactly the values that quantizer quantizes.
cudaError_t launch_quantize_append_mma(const QuantArgs& a, int d, int bits, int group,
                                       cudaStream_t stream, bool* supported);
// The per-channel key quantizer on the same tensor-core pipeline: one
// 128-token block of one head per tile.
cudaError_t launch_quantize_key_channels_mma(const QuantArgs& a, int d, int bits,
                                             cudaStream_t stream, bool* supported);
cudaError_t launch_quant_wait_selftest(unsigned long long limit_ns, int* status,
                                      cudaStream_t stream);
cudaError_t launch_rotate_mma_f32(const uint16_t* x, long long rows, int d,
                                  const uint32_t sign_bits[4], float* out, int* status,
                                  int* bounds_site, unsigned long long wait_limit_ns,
                                  cudaStream_t stream);

// Attention ---------------------------------------------------------------

struct AttnLaunch {
  // cache
  const uint8_t* k_codes;
  const uint8_t* v_codes;
  const uint32_t* k_sz;
  const uint32_t* v_sz;
  int n_s;   // valid cached tokens per head
  int cap;
  // queries: rotated FP16 (hi and lo parts, workspace) and original BF16
  const uint16_t* q_rot;
  const uint16_t* q_rot_lo;
  const uint16_t* q_orig;
  // current chunk: original BF16 keys, rotated FP16 values (workspace)
  const uint16_t* k_cur;
  const uint16_t* v_rot;
  int n_q, n_r, bh;
  float scale;
  int corr;
  int precise_query;
  int staged_words;   // KVQ_FLAG_STAGED_WORDS: cached packed words staged by TMA
  int mass_only;
  uint16_t* out;
  float* p_s;
  float* p_r;
  uint32_t sign_bits[4];
  unsigned long long wait_limit_ns;
  // key-range split (splits > 1): partial results, then a merge kernel
  int splits, tiles_per_split;
  float* o_part;    // [splits][bh][n_q][d] fp32
  float* st_part;   // [splits][bh][n_q][3] fp32
  // per-channel keys (key_mode = KVQ_KEYS_PER_CHANNEL): cached tile t is key
  // block t % bpc of chunk slot t / bpc; n_ct cached tiles; kch_c [bh][n_ct]
  // [n_q] fp32 workspace for the per-(row, tile) correction
  int key_mode, chunk, bpc, kblk_per_head, n_ct;
  float* kch_c;
  int* status;      // device status word, set by launch_attention
  int* bounds_site; // checked build's site word, set by launch_attention
  // kernels (attention_shape): kModeOneCta / kModePair / kModeAuto; with
  // kModeAuto the per-head maxima of ||q'||^2 and of the key-norm bound
  // (workspace, [bh] each) that pick each head's kernel
  int mode;
  const float* qn2;
  const float* kn2;
};

// cached key tiles of a window of n_s tokens: 128-token tiles, or with
// per-channel keys the key blocks of each chunk slot
inline int cached_tiles(int key_mode, int n_s, int chunk, int bpc) {
  if (key_mode != KVQ_KEYS_PER_CHANNEL) return (n_s + 127) / 128;
  const int full = n_s / chunk;
  return full * bpc + (n_s - full * chunk + 127) / 128;
}

// Key-range split of the attention grid.  One attention CTA fills an SM
// (its shared memory allows no second one), so a launch of n CTAs runs in
// ceil(n / sms) waves.  Splitting every (head, query block) into ranges of
// `per` key tiles costs about ceil(ctas * ranges / sms) * (per + kCtaFixed)
// tile-times (kCtaFixed: a CTA's set-up, pipeline fill and epilogue), plus
// the partial results written and merged (ranges * rows * (4d + 12) bytes,
// twice, at kBytesPerTileTime).  The split taken is the cheapest, the
// smallest on ties, with at least two tiles per range and at most
// min(64, max_splits) ranges; it helps small grids (few heads or query rows)
// and grids whose last wave is mostly empty.
constexpr int kCtaFixed = 2;
constexpr double kBytesPerTileTime = 12e6;

// CTAs of one unsplit launch: one per (head, block of rows_per_cta query
// rows), or with SM pairs two per block of 2 * rows_per_cta rows
inline long long attention_ctas(long long bh, int n_q, int rows_per_cta, bool pair) {
  if (!pair) return bh * ((n_q + rows_per_cta - 1) / rows_per_cta);
  return 2 * bh * ((n_q + 2 * rows_per_cta - 1) / (2 * rows_per_cta));
}

// cost: when not null, the estimated time of the chosen plan in tile-times
// (of a CTA of this shape)
inline void attention_split(long long bh, int n_q, int n_ct, int n_r, int d, int rows_per_cta,
                            int sms, int max_splits, int* splits, int* tiles_per_split,
                            bool pair = false, double* cost = nullptr) {
  const int n_t = n_ct + (n_r + 127) / 128;
  *splits = 1;
  *tiles_per_split = n_t > 0 ? n_t : 1;
  const long long ctas = attention_ctas(bh, n_q, rows_per_cta, pair);
  const long long waves1 = sms > 0 ? (ctas + sms - 1) / sms : 1;
  double best = (double)waves1 * (n_t + kCtaFixed);
  if (cost != nullptr) *cost = best;
  if (n_t < 4 || ctas <= 0 || sms <= 0 || max_splits < 2) return;
  int lim = n_t / 2;
  if (lim > 64) lim = 64;
  if (lim > max_splits) lim = max_splits;
  const double row_bytes = 2.0 * (double)bh * n_q * (4.0 * d + 12.0);
  for (int sp = 2; sp <= lim; ++sp) {
    const int per = (n_t + sp - 1) / sp;
    const int used = (n_t + per - 1) / per;
    const double c = (double)((ctas * used + sms - 1) / sms) * (per + kCtaFixed) + 1.0 +
                     used * row_bytes / kBytesPerTileTime;
    if (c < best) {
      best = c;
      *splits = used;
      *tiles_per_split = per;
    }
  }
  if (cost != nullptr) *cost = best;
}

// Kernels of one attention call (head_dim, key mode and correction decide):
//   kModeOneCta  the one-CTA kernel alone: two query tiles per CTA, or one
//                with the precise-query split or the exact correction;
//   kModePair    the SM-pair kernel alone (kvq_attn_pair.cuh: head_dim 128,
//                per-token keys, Taylor term or none) with the precise-query
//                split, two query tiles per CTA;
//   kModeAuto    both, each (batch, head) run by one of them: heads whose
//                FP16 query rounding can move the masses noticeably take the
//                pair kernel with the precise split, the others the one-CTA
//                kernel (the choice is made on the GPU from per-head norms,
//                see kPreciseSelect).
// Both kernels hold 256 query rows per SM and share one key-range split.
enum : int { kModeOneCta = 0, kModePair = 1, kModeAuto = 2 };

// Per-head choice of the precise-query split in kModeAuto.  A rotated query
// q' carries one FP16 rounding per channel (|dq_c| <= 2^-11 |q'_c|), so a
// cached score moves by scale * dq . k' and the masses by a fraction of
// that.  The GPU evaluates, per (batch, head),
//   e = scale * 2^-12 * max_j ||q'_j|| * B,
//   B^2 = max over cached keys of sum_g group * (max(|z_g|, 2^bits-1-z_g) D_g)^2
// (an upper bound of ||k_hat'||^2 from the keys' steps and zero points), and
// takes the precise split when e >= kPreciseSelect.  This is an empirical
// criterion: on the synthetic workloads e is at most 0.042 where keys are
// Gaussian with outlier channels (mass error of the FP16 query <= 3.8e-4)
// and at least 0.27 where keys are Student-t(3) (mass error up to 2.8e-3
// without the split); the threshold sits between them.  Callers that want
// the split regardless pass KVQ_FLAG_PRECISE_QUERY.
constexpr float kPreciseSelect = 0.08f;

struct AttnShape {
  int mode;             // kModeOneCta, kModePair or kModeAuto
  int nq;               // one-CTA kernel: query tiles of 128 rows per CTA
  int splits, tiles_per_split;
};
inline AttnShape attention_shape(long long bh, int n_q, int n_ct, int n_r, int d, int mode,
                                 bool one_tile, int sms, int max_splits) {
  AttnShape sh{mode, mode == kModeOneCta && one_tile ? 1 : 2, 1, 1};
  // kModeAuto plans for the one-CTA grid (the pair kernel runs the same
  // ranges over its own grid)
  attention_split(bh, n_q, n_ct, n_r, d, 128 * sh.nq, sms, max_splits, &sh.splits,
                  &sh.tiles_per_split, mode == kModePair);
  return sh;
}

kvq_status launch_attention(const AttnLaunch& a, int d, int bits, int group,
                            cudaStream_t stream);
// device address of the attention status word (first in-kernel error since
// it was last read) in the current device's current context, or null
int* status_ptr();
// counts a kernel launch of this library while kvq_profile_begin/end records
void note_launch();
int* bounds_site_ptr();
kvq_status read_and_clear_bounds_site(int* line);
// the attention kernels of the exact correction and of per-channel keys,
// built in translation units of their own (a.status must be set)
kvq_status launch_attention_exact(const AttnLaunch& a, int d, int bits, int group,
                                  cudaStream_t stream);
kvq_status launch_attention_kch(const AttnLaunch& a, int d, int bits, int group,
                                cudaStream_t stream);
// the SM-pair kernel with the precise-query split (head_dim 128; a.status
// must be set); select: 0 every head, +1 only the heads kModeAuto gives it
kvq_status launch_attention_pair(const AttnLaunch& a, int bits, int group, int select,
                                 cudaStream_t stream);
// kModeAuto: per (batch, head) the two maxima of kPreciseSelect -- kn2[bh]
// the bound B^2 over the head's cached keys, qn2[bh] = max_j ||q_j||^2 over
// its queries (= ||q'_j||^2: the rotation is orthogonal) -- from the cache's
// steps and zero points and the BF16 queries q [bh][n_q][128].
cudaError_t launch_select_norms(const uint32_t* k_sz, const uint16_t* q, int bh, int n_s, int cap,
                                int n_q, int g, int group, int bits, float* kn2, float* qn2,
                                cudaStream_t stream);
kvq_status read_and_clear_attention_status(int* status);
cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t stream);

}  // namespace kvq
