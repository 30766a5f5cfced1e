/*
 * kvq.h -- C ABI of libkvq: Jensen-bias-corrected low-bit KV-cache chunk
 * attention for NVIDIA GB300 (sm_103a).
 *
 * Method: "Quantized Keys Steal Attention: Bias Correction for KV-Cache
 * Compression in Video Diffusion" (Tuncer, Becker, Pfeil).  Each entry point
 * names the passage that defines the operation it runs.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Tensors are contiguous, row-major, BF16 stored as raw uint16_t bits:
 *   [batch][heads][tokens][head_dim].  All pointers to tensor data are DEVICE
 *   pointers of the current CUDA device, at least 16-byte aligned.
 * - The caller owns every buffer (cache, inputs, outputs, workspace).  No
 *   entry point allocates or frees memory.
 * - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *   void*, NULL = the legacy default stream).  Argument errors are detected on
 *   the host and returned before anything is launched; a failed launch returns
 *   KVQ_ERR_CUDA.  Faults detected inside a kernel (a bounded wait that ran
 *   out) are recorded in a device status word read by
 *   kvq_last_device_status().
 * - Inputs must be finite.
 * - FP16 operand range.  The attention's tensor-core operands are FP16, so
 *   the call checks on the GPU, as it runs, that they stay finite:
 *     rotated queries and current-chunk values |x'| < 65504 (with
 *     KVQ_KEYS_PER_CHANNEL and KVQ_CORR_TAYLOR the rotated query |q'| < 2047,
 *     which the correction pre-pass squares);
 *     cached key step sizes D with (16 + o) D < 65504, o = 0 for INT2 and 8
 *     for INT4 (INT2: D < 4094, INT4: D < 2729);
 *     cached values (|z| + 2^bits - 1) D < 65504 per group.
 *   A call that meets an operand outside these limits still runs to the end,
 *   records KVQ_ERR_RANGE in the device status word (see
 *   kvq_last_device_status) and its outputs are not valid.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,  /* null pointer, bad size or mode               */
  KVQ_ERR_UNSUPPORTED = 2,  /* head_dim / bits / group not built            */
  KVQ_ERR_CAPACITY = 3,     /* append refused by the window rules           */
  KVQ_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed            */
  KVQ_ERR_TIMEOUT = 5,      /* a kernel's bounded wait ran out              */
  KVQ_ERR_ALIGNMENT = 6,    /* a pointer is not 16-byte aligned             */
  KVQ_ERR_TOO_LARGE = 7,    /* needs more than the built-in scratch holds   */
  KVQ_ERR_RANGE = 8,        /* an operand left the FP16 range (see below)   */
  KVQ_ERR_BOUNDS = 9        /* checked build only: an index left its buffer */
} kvq_status;

/* Correction applied to cached-key scores before the softmax. */
typedef enum {
  KVQ_CORR_NONE = 0,   /* plain quantized attention (the ablation)         */
  KVQ_CORR_TAYLOR = 1, /* second-order Jensen-bias correction              */
  KVQ_CORR_EXACT = 2   /* the exact log-moment of uniform noise (below)    */
} kvq_corr;

/*
 * Attention flags.
 * KVQ_FLAG_PRECISE_QUERY: the rotated query, a tensor-core operand of the
 *   cached-segment scores, is split into FP16 high and low parts and both are
 *   contracted with the cached keys (one extra QK^T pass on cached tiles),
 *   and the correction's factors get the same split, for every (batch,
 *   head).  Without the flag a rotated query carries one FP16 rounding
 *   (2^-11 relative), which moves a score by ~2^-12 of scale * |q'| |k'|:
 *   below 1e-3 on the attention masses for moderate keys, but not for keys
 *   with extreme outliers (scores of order 100).  So without the flag, for
 *   head_dim 128 with per-token keys and the Taylor term or none, the
 *   library decides per (batch, head), on the GPU and without a host
 *   synchronization: a head takes the split when
 *     scale * 2^-12 * max_j ||q'_j|| * max_i B_i >= 0.08,
 *     B_i^2 = sum_g group * (max(|z_ig|, 2^bits - 1 - z_ig) D_ig)^2
 *   (B_i bounds ||k_hat'_i|| from the cached key's steps and zero points).
 *   The threshold is empirical: it separates Gaussian keys with outlier
 *   channels (mass error <= 4e-4 without the split) from Student-t(3) keys
 *   (up to 2.8e-3).  The other configurations take the split only with the
 *   flag.  No counterpart in the paper.
 */
#define KVQ_FLAG_PRECISE_QUERY 1
/*
 * KVQ_FLAG_NO_KV_SPLIT: when batch * heads * query tiles do not fill the GPU
 * (small chunks), the attention divides the key tiles among several CTAs
 * per query tile and merges their partial softmax states (an implementation
 * choice of this library, not part of the method).  This flag turns the
 * split off (for comparisons).
 */
#define KVQ_FLAG_NO_KV_SPLIT 2
/*
 * KVQ_FLAG_ONE_CTA: with head_dim 128, per-token keys and no correction or
 * the Taylor term, the library chooses per head whether the rotated query
 * needs the precise split, and runs those heads on SM pairs (two CTAs of a
 * cluster share each key tile's dequantization and one M = 256 tensor-core
 * MMA).  This flag turns the choice off: every head runs on the one-CTA
 * kernel without the split (for comparisons; KVQ_FLAG_PRECISE_QUERY still
 * forces the split).  An implementation choice of this library.
 */
#define KVQ_FLAG_ONE_CTA 4
/*
 * KVQ_FLAG_STAGED_WORDS: for head_dim 128, INT2 groups of 32 and the heads
 * that run without the precise split, the one-CTA kernel stages each cached
 * tile's packed codes and (step, zero) words into shared memory with TMA
 * bulk copies, one tile ahead, instead of loading them per thread.  Same
 * results (bit for bit); measured ~7 % slower on GB300, so off by default.
 * Other geometries ignore it.  An implementation choice of this library.
 */
#define KVQ_FLAG_STAGED_WORDS 8

/*
 * Key quantization scheme of a cache (kvq_cache.key_mode).
 * KVQ_KEYS_PER_TOKEN: keys like values, per token and group of `group`
 *   channels (paper section 3, "Quantization granularity").
 * KVQ_KEYS_PER_CHANNEL: keys per channel over blocks of KVQ_KEY_BLOCK tokens,
 *   the blocks counted from the first token of every appended chunk (the
 *   last block of a chunk may be shorter); values stay per token and group.
 *   This is the KIVI-style per-channel key quantization the paper's section 2
 *   lists among the schemes its correction is orthogonal to.  The correction
 *   keeps its form with one channel per group:
 *   b_ij = scale^2 / 24 * sum_c q'_{j,c}^2 * D_{c,blk(i)}^2 (TAYLOR), or the
 *   exact sum_c log(sinh a_c / a_c) with a_c = scale/2 |q'_{j,c}| D_{c,blk(i)}.
 *   The attention adds a per-(query row, key block) table to the workspace
 *   (see kvq_workspace_bytes); with TAYLOR its tensor-core pre-pass needs
 *   rotated query values |q'| < 2047.
 */
#define KVQ_KEYS_PER_TOKEN 0
#define KVQ_KEYS_PER_CHANNEL 1
#define KVQ_KEY_BLOCK 128

/*
 * Quantized sliding-window KV cache (paper section 1: the current chunk
 * attends to the last n cached chunks; section 3 "Integer quantization",
 * Eq. (1), and "Quantization granularity": per-token groups of `group`
 * channels with their own step size and zero point).
 *
 * Geometry (set by the caller, checked by every call):
 *   head_dim in {64, 128}; bits in {2, 4}; group in {32, 64}, group <= head_dim;
 *   capacity = chunk_tokens * n_chunks tokens per (batch, head).
 * Ring state (owned by the library, updated by kvq_quantize_append):
 *   len       valid tokens; attention reads tokens [0, len) of every head;
 *   head_slot chunk slot the next append writes.
 * Rotation: sign_bits[c / 32] bit (c % 32) set means sigma_c = -1 in the
 *   randomized Hadamard rotation H = (1/sqrt(d)) * Sylvester(d) * diag(sigma)
 *   (paper section 3 "Hadamard rotation").  Host values.
 * Device buffers (caller-allocated; sizes from kvq_cache_bytes):
 *   k_codes, v_codes  uint8  [batch][heads][capacity][head_dim * bits / 8]
 *       packed codes: little-endian 32-bit words; INT2 channel 16w + 2k + h
 *       at bits [2k + 16h, +2) of word w; INT4 channel 8w + 2k + h at bits
 *       [4k + 16h, +4).
 *   k_sz, v_sz        bf16   [batch][heads][capacity][head_dim / group][2]
 *       (step size, zero point) per token and group; the zero point is an
 *       integer stored as BF16.
 *   With key_mode = KVQ_KEYS_PER_CHANNEL, k_sz instead holds
 *       bf16 [batch][heads][n_chunks][ceil(chunk_tokens / KVQ_KEY_BLOCK)]
 *       [head_dim][2]: (step size, zero point) per key block and channel
 *       (block b of slot s covers tokens s * chunk_tokens + [128 b, 128 b +
 *       128)); k_codes keeps the per-token layout above.
 * key_mode: KVQ_KEYS_PER_TOKEN (0) or KVQ_KEYS_PER_CHANNEL (1).
 */
typedef struct kvq_cache {
  int32_t batch, heads, head_dim, bits, group;
  int32_t chunk_tokens, n_chunks;
  int32_t len, head_slot;
  uint32_t sign_bits[4];
  uint8_t *k_codes, *v_codes;
  uint16_t *k_sz, *v_sz;
  int32_t key_mode;
} kvq_cache;

/* Human-readable name of a status code (static string, never NULL). */
const char *kvq_status_string(kvq_status s);

/* Library ABI version (increments on any change of this header's ABI). */
int32_t kvq_abi_version(void);

/*
 * Bytes of ONE codes buffer and of the larger of the two (step, zero)
 * buffers for this geometry (k and v each need a codes buffer of
 * codes_bytes; sz_bytes is enough for either of k_sz and v_sz).  Returns
 * KVQ_ERR_INVALID_ARG / KVQ_ERR_UNSUPPORTED for a bad geometry.  Host only;
 * no CUDA call.
 */
kvq_status kvq_cache_bytes(const kvq_cache *cache, size_t *codes_bytes,
                           size_t *sz_bytes);

/*
 * Exact bytes of k_sz and of v_sz (they differ with KVQ_KEYS_PER_CHANNEL).
 * Host only; no CUDA call.
 */
kvq_status kvq_cache_meta_bytes(const kvq_cache *cache, size_t *k_sz_bytes,
                                size_t *v_sz_bytes);

/*
 * Quantize-append one chunk (paper section 3: Hadamard rotation, then
 * Eq. (1) per token and group; Figure 1 caption: keys AND values, QuaRot +
 * RTN).  k_new, v_new: BF16 [batch][heads][n_new][head_dim] device.
 * Per row: x' = fl(1/sqrt(d)) * S with S = Sylvester(d) diag(sigma) x summed
 * in fp32 by the tensor cores (every product exact; the summation order is
 * the hardware's, deterministic: a row gives the same bits wherever it sits
 * in the input; kvq_rotate's fp32 output returns exactly these values); per
 * group mn/mx; D = bf16((mx - mn) / (2^bits - 1)) (constant group:
 * D = bf16(|mn|), or 1); z = bf16(rint(-mn / D)); code =
 * clamp(rint(x' / D) + z, 0, 2^bits-1) (IEEE fp32, ties to even).  Writes
 * slot `head_slot` (tokens [head_slot * chunk_tokens, + n_new)).  With
 * KVQ_KEYS_PER_CHANNEL the keys take the same steps per channel over each
 * block of KVQ_KEY_BLOCK tokens of the chunk (mn/mx over the block's values
 * of that channel), on x' from the fast Walsh-Hadamard transform
 * (butterflies in the order h = 1, 2, ..., d/2 in fp32, then times
 * fl(1/sqrt(d))); the values stay per token as above.
 * Window rules: 0 <= n_new <= chunk_tokens (0 is a no-op); while the cache is
 * not full every earlier slot must be full (a partial chunk can only be the
 * last one appended); once full only whole chunks overwrite the oldest slot.
 * Otherwise KVQ_ERR_CAPACITY and nothing changes.  On success updates
 * cache->len and cache->head_slot (host side, no synchronization).
 */
kvq_status kvq_quantize_append(kvq_cache *cache, const uint16_t *k_new,
                               const uint16_t *v_new, int32_t n_new,
                               void *stream);

/*
 * Workspace bytes kvq_attention_corrected / kvq_attention_mass need for n_q
 * queries and n_r current-chunk tokens: the rotated query (FP16 high and low
 * parts), the rotated current values (FP16), when the launch would not fill
 * the current device the partial results of the key-range split (fp32), and
 * with per-channel keys one fp32 per query row and cached key block (the
 * block's zero-point term minus the correction), and two floats per (batch,
 * head) (the per-head choice of the precise-query split, below).  Depends on
 * the current device's SM count.  0 on a bad geometry.
 */
size_t kvq_workspace_bytes(const kvq_cache *cache, int32_t n_q, int32_t n_r);

/*
 * Corrected chunk attention (paper abstract and section 1; Figure 3 caption).
 * Queries q [batch][heads][n_q][d] of the current chunk attend over the
 * dequantized cached window (tokens [0, cache->len), rotated basis) and the
 * unquantized current chunk k_cur, v_cur [batch][heads][n_r][d].  No mask.
 *   cached score  s_ij = scale * q'_j . k_hat'_i - b_ij,
 *   b_ij = scale^2 / 24 * sum_g ||q'_{j,g}||^2 * D_{i,g}^2   (corr = TAYLOR;
 *          0 for corr = NONE) -- the second-order Jensen-bias correction;
 *   corr = EXACT: b_ij = sum_c log(sinh(a_c) / a_c), a_c = scale/2 *
 *          |q'_{j,c}| * D_{i,g(c)} -- log E[exp(delta)] for independent
 *          uniform rounding noise on every rotated key channel, of which the
 *          TAYLOR term is the leading a^2/6 part (Figure 3 caption; the
 *          paper's correction is the Taylor one, this mode measures what the
 *          truncation leaves out).  Evaluated in fp32: a power series in the
 *          key's step size against per-row moments of the query while every
 *          a_c of a group is <= 1, per channel otherwise.  Runs with one
 *          query tile per CTA and costs several times the TAYLOR mode;
 *   current score s_ij = scale * q_j . k_i on the unrotated BF16 inputs
 *          (exact products, fp32 accumulation);
 *   one softmax over both segments; out = sum_i p_ij v_i in the ORIGINAL
 *   basis (cached values un-rotated).
 * flags: any combination of KVQ_FLAG_PRECISE_QUERY, KVQ_FLAG_NO_KV_SPLIT,
 * KVQ_FLAG_ONE_CTA and KVQ_FLAG_STAGED_WORDS (0 for none).
 * out: BF16 [batch][heads][n_q][d] device (required).  p_s, p_r: optional
 * (NULL to skip) fp32 [batch][heads][n_q] device: the attention masses of the
 * cached block and of the current chunk per query row (Figure 2 caption).
 * workspace: device, >= kvq_workspace_bytes(cache, n_q, n_r) bytes, 16-byte
 * aligned; its contents are scratch (the rotated query as FP16 high and low
 * parts and the rotated current values in FP16: tensor-core operands; the
 * key-range split's partial results).
 * The FP16 operand limits of the conventions above apply (KVQ_ERR_RANGE in
 * the device status word when broken).  Requires cache->len + n_r >= 1 when
 * n_q > 0.  n_q == 0 is a no-op.
 */
kvq_status kvq_attention_corrected(const kvq_cache *cache, const uint16_t *q,
                                   const uint16_t *k_cur, const uint16_t *v_cur,
                                   int32_t n_q, int32_t n_r, float scale,
                                   int32_t corr, int32_t flags, void *workspace,
                                   size_t workspace_bytes, uint16_t *out,
                                   float *p_s, float *p_r, void *stream);

/*
 * Attention masses only (paper Figure 2 caption and section 1: P_S of the
 * cached block, P_R of the current chunk; P_S + P_R = 1 per row), with the
 * same scores as kvq_attention_corrected.  v_cur is not read.  p_s, p_r:
 * fp32 [batch][heads][n_q] device (both required).
 */
kvq_status kvq_attention_mass(const kvq_cache *cache, const uint16_t *q,
                              const uint16_t *k_cur, int32_t n_q, int32_t n_r,
                              float scale, int32_t corr, int32_t flags,
                              void *workspace,
                              size_t workspace_bytes, float *p_s, float *p_r,
                              void *stream);

/*
 * The rotation alone (paper section 3 "Hadamard rotation"), for checking:
 * x' = H x per row of x [rows][d] BF16 device, either
 *   out_f32: fp32 [rows][d], the tensor-core product -- exactly the values
 *            kvq_quantize_append quantizes per token; or
 *   out_f16: FP16 [rows][d], the fast Walsh-Hadamard transform in fp32
 *            (butterflies h = 1, 2, ..., d/2, then times fl(1/sqrt(d)))
 *            rounded to FP16 -- exactly the tensor-core operands the
 *            attention kernels read for q and the current chunk's values
 *            (the current keys enter unrotated, in BF16).
 * The two fp32 evaluations differ by rounding only (a few units of 2^-24
 * relative to sum |x|).  Exactly one of out_f32 / out_f16 must be non-NULL.
 * d in {64, 128}.
 */
kvq_status kvq_rotate(const uint16_t *x, int64_t rows, int32_t d,
                      const uint32_t sign_bits[4], float *out_f32,
                      uint16_t *out_f16, void *stream);

/*
 * Synchronizes `stream`, then returns and clears the device status word of
 * the current device (KVQ_OK, or the first in-kernel error since the last
 * call: KVQ_ERR_TIMEOUT, KVQ_ERR_RANGE, or in the checked build
 * KVQ_ERR_BOUNDS).  Returns KVQ_ERR_CUDA if the synchronization failed.
 */
kvq_status kvq_last_device_status(void *stream);

/*
 * Checked build (the same sources compiled with -DKVQ_DEBUG_BOUNDS into
 * libkvq_checked.so; a debugging aid, not the product's fast path): every
 * kernel tests the indices of its global-memory accesses to the caches, the
 * inputs and the outputs against the extents the call passed, skips an
 * access that falls outside, and records KVQ_ERR_BOUNDS in the device status
 * word and the source line of the first such check in a site word.
 * Synchronizes `stream`, then stores and clears that line in *line (0 when
 * no check failed; always 0 in the regular build, whose checks compile to
 * nothing).  Returns KVQ_ERR_INVALID_ARG for a NULL line, KVQ_ERR_CUDA if
 * the synchronization or the read failed.
 */
kvq_status kvq_debug_bounds_site(int32_t *line, void *stream);
/* 1 in the checked build, 0 in the regular one. */
int32_t kvq_debug_bounds_build(void);

/*
 * Limit, in nanoseconds, of every bounded wait inside the kernels (default
 * 2e9).  Exceeding it makes the kernel record KVQ_ERR_TIMEOUT, release its
 * tensor memory and return.  Host setting, applies to later launches.  (The
 * quantizer waits for its own copies and MMAs in flight for at least 100 ms
 * before it exits, whatever the limit.)
 */
kvq_status kvq_set_wait_limit_ns(uint64_t limit_ns);

/*
 * Self-test of the bounded-wait path: two one-block kernels, one with the
 * attention kernels' wait and one with the tensor-core quantizer's, each
 * wait on a shared-memory barrier that nothing ever arrives on, for at most
 * limit_ns, then record KVQ_ERR_TIMEOUT and return.  No counterpart in the
 * paper; it exists so the error path can be exercised without faulting or
 * hanging a GPU.
 */
kvq_status kvq_selftest_wait_timeout(uint64_t limit_ns, void *stream);

/*
 * kvq_attention_corrected without a workspace argument, for callers that
 * cannot allocate device memory when they call: for instance a plugin whose
 * host process owns every byte of the device through its own pool, a
 * real-time loop that may not take the allocator's locks or its implicit
 * synchronization, or a deployment whose device-memory budget is fixed when
 * the library is loaded.  No counterpart in the paper.
 *
 * Same arguments, meaning and results as kvq_attention_corrected, minus the
 * workspace.  The scratch space comes from one fixed device buffer of
 * KVQ_NOALLOC_SCRATCH_BYTES (32 MiB) inside the library; every device that
 * loads the library holds it until the process exits.  The call is refused
 * with KVQ_ERR_TOO_LARGE, before anything is launched, when the scratch of
 * the unsplit launch for the cache's current window (the rotated query as
 * FP16 high and low parts, the rotated current values, two floats per
 * (batch, head), and with KVQ_KEYS_PER_CHANNEL one fp32 per query row and
 * cached key block) exceeds
 * KVQ_NOALLOC_SCRATCH_BYTES; when it fits, the key-range split (which needs
 * room for partial results) takes the largest number of ranges whose
 * scratch still fits, down to none.  The limit is therefore not
 * kvq_workspace_bytes(), which sizes the split for a full window.
 * - The first call on a device, and the first after the device's context
 *   changed (after cudaDeviceReset, for instance), looks up the buffer's
 *   device address in the current context (with that device current); make
 *   those calls before any stream capture.
 * - All calls share the one buffer and it keeps the previous call's contents
 *   (nothing in it needs to start at zero: each call overwrites what it
 *   reads).  Calls whose kernels overlap on the GPU -- on different streams,
 *   or from different host threads -- race on it; serialize them.
 * - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 */
#define KVQ_NOALLOC_SCRATCH_BYTES (32u << 20)
kvq_status kvq_attention_corrected_noalloc(const kvq_cache *cache, const uint16_t *q,
                                           const uint16_t *k_cur, const uint16_t *v_cur,
                                           int32_t n_q, int32_t n_r, float scale,
                                           int32_t corr, int32_t flags, uint16_t *out,
                                           float *p_s, float *p_r, void *stream);

/*
 * Instrumentation (no counterpart in the paper).  Between kvq_profile_begin
 * and kvq_profile_end the library records a pair of CUDA events around each
 * phase of a call, on the stream the call runs on: the quantize-append (one
 * kernel, two with per-channel keys), the rotation (the rotation kernel, and
 * the per-head selection pass before it in the automatic choice of the
 * precise split), the attention (its kernels and the merge of a key-range
 * split).  kvq_profile_end waits for those events and returns, per kind
 * (0 quantize-append, 1 rotation, 2 attention), the summed device time in
 * milliseconds and the number of recorded phases, then stops recording.  At
 * most 16384 phases per kind are recorded.  kvq_profile_kernel_launches
 * returns the number of kernels the library launched since the last
 * kvq_profile_begin while recording.  Process-global; not thread-safe.
 */
kvq_status kvq_profile_begin(void);
kvq_status kvq_profile_end(double ms_total[3], int32_t launches[3]);
int64_t kvq_profile_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
