"""CPU oracle for Jensen-bias-corrected low-bit KV-cache chunk attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA path (``quantized_kv_cache_quantize_gb300/csrc``).

Source: "Quantized Keys Steal Attention: Bias Correction for KV-Cache
Compression in Video Diffusion" (Tuncer, Becker, Pfeil), cited below as
"the paper", by section / equation / figure:

* section 3 "Integer quantization", Eq. (1): asymmetric round-to-nearest
  x_q = clamp(round(x / Delta) + z, 0, 2^B - 1), x_hat = (x_q - z) * Delta,
  |x_hat - x| <= Delta / 2, Delta and z chosen to cover [min, max];
* section 3 "Quantization granularity": per-token groups of g channels, each
  group with its own (Delta, z);
* section 3 "Hadamard rotation": a randomized Hadamard H (H^T H = I) applied to
  keys and queries, which preserves scores (Hq)^T (Hk) = q^T k; Figure 1's
  caption applies QuaRot + RTN to keys and values;
* Figure 3 caption, abstract and section 1: quantization noise
  delta ~ Uniform[-Delta/2, Delta/2] on a score makes E[exp(s + delta)] exceed
  exp(s) (the Jensen bias); a per-score correction b, computed from the cached
  keys' step sizes and the query norm, is subtracted before the softmax from
  cached-key scores only, with a second-order Taylor approximation;
* Figure 2 caption / section 1: the attention masses P_S (cached block) and
  P_R (current chunk);
* section 2 (related work): per-channel key quantization (KIVI) is among the
  schemes the correction is said to be orthogonal to -- the per-channel key
  mode below quantizes each key channel over blocks of 128 tokens with the
  same Eq. (1), and the correction keeps its form with one channel per group.

Everything is fp64 except the steps that are fp32 on purpose, because the
GPU reproduces them bit for bit: the code decision (``quantize_groups``) and
the butterfly rotation (``rotate_fp32``, the textbook fast Walsh-Hadamard
transform in fp32) that the attention's FP16 operands and the per-channel
key quantizer use.  The per-token quantizer rotates on the tensor cores,
which sum in an order of their own: for it ``rotation_bounds`` bounds every
fp32 summation order and ``quantize_groups_admissible`` lists every answer
Eq. (1) gives inside those bounds (one answer wherever the bounds fix it).
Where the paper is silent the readings are listed in each docstring.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, hand-worked fixtures under ``tests/golden``, brute force,
Monte-Carlo, invariants).  The magnitude of the attention-mass shift and the
end-to-end output on the synthetic workloads have no printed value in the
paper: beyond the invariants those two are "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# BF16 rounding (storage format of the step sizes, zero points and tensors)
# ---------------------------------------------------------------------------


def bf16_round(x) -> np.ndarray:
    """Round float32 values to the nearest BF16 (ties to even), returned as
    float32.  BF16 keeps the top 16 bits of an IEEE float32; finite inputs
    only."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    bits = a.view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    bits = (bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    out = (bits << np.uint64(16)).astype(np.uint32)
    return out.view(np.float32).reshape(a.shape)


def bf16_bits(x) -> np.ndarray:
    """The 16-bit pattern of float32 values that are already BF16-exact."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    return (a.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def from_bf16_bits(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


# ---------------------------------------------------------------------------
# Randomized Hadamard rotation (paper section 3, "Hadamard rotation")
# ---------------------------------------------------------------------------


def sylvester_hadamard(d: int) -> np.ndarray:
    """Sylvester construction: H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]].

    Reading: the paper names a "randomized Hadamard rotation" without its
    construction; we take the Sylvester matrix times a random sign diagonal,
    normalised by 1/sqrt(d) (the QuaRot construction it cites)."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def rotation_matrix(signs) -> np.ndarray:
    """R = (1/sqrt(d)) * H_Sylvester * diag(signs); orthogonal, so R^T R = I."""
    s = np.asarray(signs, dtype=np.float64)
    d = s.shape[0]
    return sylvester_hadamard(d) * s[None, :] / math.sqrt(d)


def rotate(x, signs) -> np.ndarray:
    """x' = R x for each row x (fp64)."""
    return np.asarray(x, dtype=np.float64) @ rotation_matrix(signs).T


def unrotate(y, signs) -> np.ndarray:
    """x = R^T y for each row y (fp64), the inverse of ``rotate``."""
    return np.asarray(y, dtype=np.float64) @ rotation_matrix(signs)


def rotate_fp32(x, signs) -> np.ndarray:
    """The rotation in fp32, as the fast Walsh-Hadamard transform.

    Steps (each a correctly rounded IEEE fp32 operation): multiply by the
    signs (exact); then for h = 1, 2, 4, ..., d/2, for every index i whose bit
    h is clear, replace (x[i], x[i+h]) by (x[i] + x[i+h], x[i] - x[i+h]);
    finally multiply by the fp32 constant fl(1/sqrt(d)).  In exact
    arithmetic this equals ``rotate``; in fp32 it fixes one rounding order,
    which the quantizer's bit-exact contract is defined on."""
    y = np.array(x, dtype=np.float32, copy=True)
    lead = y.shape[:-1]
    d = y.shape[-1]
    y = y * np.asarray(signs, dtype=np.float32)
    h = 1
    while h < d:
        v = y.reshape(*lead, d // (2 * h), 2, h)
        a = v[..., 0, :]
        b = v[..., 1, :]
        y = np.stack([a + b, a - b], axis=-2).reshape(*lead, d)
        h *= 2
    inv = np.float32(1.0 / math.sqrt(float(d)))
    return (y * inv).astype(np.float32)


# ---------------------------------------------------------------------------
# Asymmetric per-token-group quantization (paper section 3, Eq. (1))
# ---------------------------------------------------------------------------


def quantize_groups(y, bits: int, group: int):
    """Quantize fp32 rows y [..., d] per token and group of ``group`` channels.

    Returns (codes uint8 [..., d], delta float32 [..., G], zero float32
    [..., G]); delta and zero are BF16-exact (they are stored as BF16).

    Per group, in fp32:
      mn, mx   = min, max of the group            (Eq. (1): cover [min, max])
      delta    = bf16(fl((mx - mn) / (2^B - 1)))
      if delta == 0: delta = bf16(|mn|), and 1 if that is 0 too
      zero     = bf16(rint(fl(-mn / delta)) + 0)   (integer zero point)
      code     = clamp(rint(fl(y / delta)) + zero, 0, 2^B - 1)

    Readings where the paper is silent: rint rounds half to even; z is an
    integer and is not clamped (all-positive or all-negative groups need
    that); codes are computed with the stored BF16 delta and zero so that
    quantize and dequantize agree; "+ 0" turns a -0 zero point into +0; a
    constant group (delta would be 0) takes delta = |mn| so that it
    dequantizes to its own value."""
    y = np.asarray(y, dtype=np.float32)
    d = y.shape[-1]
    if d % group:
        raise ValueError("group must divide d")
    lead = y.shape[:-1]
    g_n = d // group
    yg = y.reshape(*lead, g_n, group)
    mn = yg.min(axis=-1)
    mx = yg.max(axis=-1)
    qmax = np.float32(2 ** bits - 1)
    delta = bf16_round((mx - mn) / qmax)
    fb = bf16_round(np.abs(mn))
    fb = np.where(fb == 0, np.float32(1.0), fb).astype(np.float32)
    delta = np.where(delta == 0, fb, delta).astype(np.float32)
    zero = bf16_round(np.rint((-mn) / delta) + np.float32(0.0))
    codes = np.rint(yg / delta[..., None]) + zero[..., None]
    codes = np.clip(codes, np.float32(0.0), qmax)
    return codes.astype(np.uint8).reshape(*lead, d), delta, zero


def dequantize(codes, delta, zero, group: int) -> np.ndarray:
    """x_hat = (x_q - z) * delta per group, in fp64 (Eq. (1))."""
    c = np.asarray(codes, dtype=np.float64)
    lead = c.shape[:-1]
    d = c.shape[-1]
    cg = c.reshape(*lead, d // group, group)
    out = (cg - np.asarray(zero, np.float64)[..., None]) * np.asarray(delta, np.float64)[..., None]
    return out.reshape(*lead, d)


# ---------------------------------------------------------------------------
# Per-channel key quantization over token blocks (KIVI-style; the paper's
# section 2 lists per-channel key quantization among the KV-cache schemes its
# correction is orthogonal to)
# ---------------------------------------------------------------------------

KEY_BLOCK = 128


def chunk_blocks(n_tokens: int, block: int = KEY_BLOCK):
    """[start, end) of the token blocks of one appended chunk: consecutive
    blocks of ``block`` tokens from the chunk's first token, the last one
    shorter when the chunk is not a multiple of ``block``.

    Reading: the scheme groups keys per channel along tokens; blocks restart
    at every chunk, so a chunk is quantized when it is appended and never
    again (no block spans two chunks)."""
    return [(b, min(b + block, n_tokens)) for b in range(0, n_tokens, block)]


def quantize_key_channels(y, bits: int, block: int = KEY_BLOCK):
    """Per-channel quantization of one chunk's rotated fp32 keys y [n, d]:
    for every block of tokens and every channel, Eq. (1) over that channel's
    values in the block -- the same step, zero point and rounding as
    ``quantize_groups``, with the group running along tokens instead of
    channels.  Returns (codes uint8 [n, d], delta float32 [n_blocks, d],
    zero float32 [n_blocks, d])."""
    y = np.asarray(y, dtype=np.float32)
    n, d = y.shape
    blocks = chunk_blocks(n, block)
    codes = np.empty((n, d), dtype=np.uint8)
    delta = np.empty((len(blocks), d), dtype=np.float32)
    zero = np.empty((len(blocks), d), dtype=np.float32)
    for i, (a, b) in enumerate(blocks):
        c, dl, z = quantize_groups(np.ascontiguousarray(y[a:b].T), bits, b - a)
        codes[a:b] = c.T
        delta[i] = dl[:, 0]
        zero[i] = z[:, 0]
    return codes, delta, zero


def quantize_key_channels_admissible(y_lo, y_hi, bits: int, block: int = KEY_BLOCK):
    """Every answer ``quantize_key_channels`` can give for fp32 keys y [n, d]
    with y_lo <= y <= y_hi elementwise: per block of tokens,
    ``quantize_groups_admissible`` over each channel's values in the block
    (the group running along tokens, as in ``quantize_key_channels``).
    Returns one tuple per block: delta, zero [d, 4] and code_lo, code_hi
    [d, 4, block tokens] (the block's codes transposed: channel, candidate,
    token)."""
    lo = np.asarray(y_lo, dtype=np.float32)
    hi = np.asarray(y_hi, dtype=np.float32)
    out = []
    for a, b in chunk_blocks(lo.shape[0], block):
        cd, cz, clo, chi = quantize_groups_admissible(np.ascontiguousarray(lo[a:b].T),
                                                      np.ascontiguousarray(hi[a:b].T), bits, b - a)
        out.append((cd[:, 0], cz[:, 0], clo[:, 0], chi[:, 0]))
    return out


def key_channel_token_steps(values, n_tokens: int, block: int = KEY_BLOCK) -> np.ndarray:
    """Per-token view [n, d] of per-block, per-channel values [n_blocks, d]
    (each token gets the row of its block)."""
    v = np.asarray(values)
    idx = np.array([i for i, (a, b) in enumerate(chunk_blocks(n_tokens, block)) for _ in range(a, b)],
                   dtype=np.int64)
    return v[idx]


def dequantize_key_channels(codes, delta, zero, block: int = KEY_BLOCK) -> np.ndarray:
    """x_hat = (x_q - z) * delta with each token's block's per-channel step
    and zero point, fp64 (Eq. (1))."""
    c = np.asarray(codes, dtype=np.float64)
    n = c.shape[0]
    dl = key_channel_token_steps(np.asarray(delta, np.float64), n, block)
    z = key_channel_token_steps(np.asarray(zero, np.float64), n, block)
    return (c - z) * dl


def quantize_key_chunk(x_bf16, signs, bits: int, block: int = KEY_BLOCK):
    """What one quantize-append computes for one chunk of BF16 keys [n, d]
    in the per-channel key mode: the fp32 rotation, then
    ``quantize_key_channels``.  Returns (packed codes, delta, zero, rotated
    fp32, codes)."""
    y = rotate_fp32(np.asarray(x_bf16, dtype=np.float32), signs)
    codes, delta, zero = quantize_key_channels(y, bits, block)
    return pack_codes(codes, bits), delta, zero, y, codes


# ---------------------------------------------------------------------------
# Packed code layout (a storage format of this library; the paper fixes none)
# ---------------------------------------------------------------------------


def pack_codes(codes, bits: int) -> np.ndarray:
    """Pack codes [..., d] into bytes [..., d * bits / 8].

    Little-endian 32-bit words of 32/bits codes each.  INT2: channel
    16w + 2k + h (k < 8, h < 2) sits at bits [2k + 16h, 2k + 16h + 2) of word
    w.  INT4: channel 8w + 2k + h (k < 4) sits at bits [4k + 16h, 4k + 16h + 4).
    Adjacent channel pairs thus land 16 bits apart in one word."""
    c = np.asarray(codes, dtype=np.uint32)
    lead = c.shape[:-1]
    d = c.shape[-1]
    per = 32 // bits
    half = per // 2
    cw = c.reshape(*lead, d // per, half, 2)
    words = np.zeros((*lead, d // per), dtype=np.uint32)
    for k in range(half):
        for h in range(2):
            shift = np.uint32(bits * k + 16 * h)
            words |= cw[..., k, h] << shift
    return np.ascontiguousarray(words.astype("<u4")).view(np.uint8).reshape(*lead, d * bits // 8)


def unpack_codes(packed, bits: int, d: int) -> np.ndarray:
    p = np.ascontiguousarray(np.asarray(packed, dtype=np.uint8))
    lead = p.shape[:-1]
    words = p.view("<u4").astype(np.uint32).reshape(*lead, -1)
    per = 32 // bits
    half = per // 2
    mask = np.uint32(2 ** bits - 1)
    out = np.zeros((*lead, d // per, half, 2), dtype=np.uint8)
    for k in range(half):
        for h in range(2):
            out[..., k, h] = (words >> np.uint32(bits * k + 16 * h)) & mask
    return out.reshape(*lead, d)


def quantize_rows(x_bf16, signs, bits: int, group: int):
    """What one quantize-append computes for rows of BF16 values x [..., d]:
    the fp32 rotation, then the per-group quantizer.  Returns
    (packed codes, delta, zero, rotated fp32, codes)."""
    y = rotate_fp32(np.asarray(x_bf16, dtype=np.float32), signs)
    codes, delta, zero = quantize_groups(y, bits, group)
    return pack_codes(codes, bits), delta, zero, y, codes


# ---------------------------------------------------------------------------
# The rotation known to within a rounding bound, and every answer Eq. (1)
# can give inside it.  For an fp32 rotation whose summation order is not
# fixed (a tensor-core product sums the d exact products sigma_k H[n][k] x_k
# in an order and with internal rounding of the hardware's choosing) the
# codes are not one value but a small set; away from rounding boundaries
# the set has one element.
# ---------------------------------------------------------------------------


def _round32(v, up: bool) -> np.ndarray:
    """fp64 values rounded to fp32 toward +inf (up) or toward -inf."""
    v = np.asarray(v, dtype=np.float64)
    r = v.astype(np.float32)
    if up:
        return np.where(r.astype(np.float64) < v, np.nextafter(r, np.float32(np.inf)), r)
    return np.where(r.astype(np.float64) > v, np.nextafter(r, np.float32(-np.inf)), r)


def _lsb_exponent(x) -> np.ndarray:
    """For fp32 values: q with x an odd multiple of 2^q (a large q for 0)."""
    m, e = np.frexp(np.asarray(x, dtype=np.float64))      # x = m 2^e, 0.5 <= |m| < 1
    mi = np.abs(m * 2.0 ** 24).astype(np.int64)              # 24-bit integer significand
    tz = np.zeros_like(mi)
    nz = mi != 0
    low = mi[nz] & -mi[nz]                                   # lowest set bit
    tz[nz] = np.log2(low.astype(np.float64)).astype(np.int64)
    q = e.astype(np.int64) - 24 + tz
    return np.where(nz, q, np.int64(1 << 20))


def rotation_bounds(x, signs):
    """Bounds [y_lo, y_hi] (fp32, elementwise) on any fp32 rotation of rows
    x [..., d] computed as y = fl(S * fl(1/sqrt(d))), S an fp32 sum of the d
    exact products sigma_k Sylvester(d)[n][k] x_k taken in any order, each
    addition rounded to nearest or toward zero.

    Bound on the sum (recursive summation, Higham, "Accuracy and Stability
    of Numerical Algorithms", section 4.2): |S - sum| <= gamma_{d-1} *
    sum_k |x_k|, gamma_n = n u / (1 - n u), u = 2^-23 (one unit of the 24-bit
    significand, which covers truncation as well as rounding to nearest).
    The bound is 0 for a row whose values are all multiples of 2^q with
    sum_k |x_k| <= 2^(24 + q): every partial sum of such a row is an fp32
    number, so every order gives the exact sum.  The exact sums are formed in
    fp64 (exact for such rows; otherwise their own error, at most
    d 2^-53 sum |x|, is added to the bound).  Then S lies in [RU(lo), RD(hi)]
    and the multiply is monotone."""
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[-1]
    s = np.asarray(signs, dtype=np.float64)
    exact_sum = x.astype(np.float64) @ (sylvester_hadamard(d) * s[None, :]).T   # [..., d]
    abs_sum = np.abs(x.astype(np.float64)).sum(axis=-1, keepdims=True)
    n = d - 1
    u = 2.0 ** -23
    gamma = n * u / (1.0 - n * u)
    q = _lsb_exponent(x).min(axis=-1, keepdims=True)
    on_grid = abs_sum <= np.ldexp(1.0, (24 + np.minimum(q, 990)).astype(np.int64))
    eps = np.where(on_grid, 0.0, gamma * abs_sum + d * 2.0 ** -53 * abs_sum)
    s_lo = _round32(exact_sum - eps, up=True).astype(np.float64)
    s_hi = _round32(exact_sum + eps, up=False).astype(np.float64)
    inv = np.float64(np.float32(1.0 / math.sqrt(float(d))))
    return (s_lo * inv).astype(np.float32), (s_hi * inv).astype(np.float32)


def _step_of(mn, mx, qmax):
    """Eq. (1)'s BF16 step for one (min, max) pair, as quantize_groups; and
    whether the constant-group rule (step 0 -> |min|, or 1) decided it."""
    delta = bf16_round((mx - mn) / qmax)
    fb = bf16_round(np.abs(mn))
    fb = np.where(fb == 0, np.float32(1.0), fb).astype(np.float32)
    return np.where(delta == 0, fb, delta).astype(np.float32), delta == 0


def _zero_of(mn, delta):
    return bf16_round(np.rint((-np.asarray(mn, np.float32)) / delta) + np.float32(0.0))


def quantize_groups_admissible(y_lo, y_hi, bits: int, group: int):
    """Every answer quantize_groups can give for fp32 rows y with
    y_lo <= y <= y_hi elementwise.

    Each step of quantize_groups is monotone given the ones before it: the
    group's min and max in the values; the fp32 subtraction, the fp32
    division by 2^B - 1 and the BF16 rounding in the span; the zero point
    (decreasing) in the min for a fixed step; a code in its value for a fixed
    step and zero point.  So the step lies between its values at the
    smallest span (min_hi, max_lo) and the largest (min_lo, max_hi); for each
    of those two steps the zero point between its values at min_hi and
    min_lo; for each (step, zero) pair a code between its values at y_lo and
    y_hi.  Returns four candidates per group: delta, zero [..., G, 4] and
    code_lo, code_hi [..., G, 4, group] (uint8).  Raises ValueError where the
    bounds are too wide for that enumeration (steps or zero points more than
    one representable value apart, or a group that may or may not be
    constant)."""
    lo = np.asarray(y_lo, dtype=np.float32)
    hi = np.asarray(y_hi, dtype=np.float32)
    if np.any(lo > hi):
        raise ValueError("y_lo > y_hi")
    d = lo.shape[-1]
    lead = lo.shape[:-1]
    g_n = d // group
    lo_g = lo.reshape(*lead, g_n, group)
    hi_g = hi.reshape(*lead, g_n, group)
    mn_lo, mn_hi = lo_g.min(axis=-1), hi_g.min(axis=-1)
    mx_lo, mx_hi = lo_g.max(axis=-1), hi_g.max(axis=-1)
    qmax = np.float32(2 ** bits - 1)
    if group == 1:
        # one value: its min and max are the same number, the span is 0
        d_small, c_small = _step_of(mn_hi, mn_hi, qmax)
        d_large, c_large = _step_of(mn_lo, mn_lo, qmax)
    else:
        d_small, c_small = _step_of(mn_hi, np.maximum(mx_lo, mn_hi), qmax)
        d_large, c_large = _step_of(mn_lo, mx_hi, qmax)
    if np.any(c_small != c_large) or np.any(c_small & (mn_lo < 0) & (mn_hi > 0)):
        raise ValueError("a group may or may not be constant within the bounds")
    # (a constant group's step |min| may come out in either order)
    d_lo, d_hi = np.minimum(d_small, d_large), np.maximum(d_small, d_large)
    next_bf16 = from_bf16_bits((bf16_bits(d_lo).astype(np.uint32) + 1).astype(np.uint16))
    if np.any(d_hi > next_bf16):
        raise ValueError("steps more than one BF16 value apart")
    deltas, zeros = [], []
    for dl in (d_small, d_large):
        z_a = _zero_of(mn_hi, dl)   # largest min: smallest zero point
        z_b = _zero_of(mn_lo, dl)
        if np.any(z_b - z_a > 1):
            raise ValueError("zero points more than one apart")
        for z in (z_a, z_b):
            deltas.append(dl)
            zeros.append(z)
    delta = np.stack(deltas, axis=-1)                        # [..., G, 4]
    zero = np.stack(zeros, axis=-1)

    def codes(y, dl, z):
        c = np.rint(y / dl[..., None]) + z[..., None]
        return np.clip(c, np.float32(0.0), qmax).astype(np.uint8)

    code_lo = np.stack([codes(lo_g, delta[..., i], zero[..., i]) for i in range(4)], axis=-2)
    code_hi = np.stack([codes(hi_g, delta[..., i], zero[..., i]) for i in range(4)], axis=-2)
    return delta, zero, code_lo, code_hi


# ---------------------------------------------------------------------------
# Jensen-bias correction (paper: abstract, section 1, Figure 3 caption)
# ---------------------------------------------------------------------------


def group_sq_norms(q_rot, group: int) -> np.ndarray:
    """n_{j,g} = ||q'_{j,g}||^2 per query row and channel group (fp64)."""
    q = np.asarray(q_rot, dtype=np.float64)
    lead = q.shape[:-1]
    d = q.shape[-1]
    return (q.reshape(*lead, d // group, group) ** 2).sum(axis=-1)


def jensen_bias_taylor(q_rot, delta, scale: float, group: int) -> np.ndarray:
    """Second-order correction b_ij = Var[delta_ij] / 2 for queries q'_j
    [Nq, d] (rotated) and cached keys with steps delta_{i,g} [Ns, G].

    The score noise is delta_ij = scale * q'_j . eps_i with independent
    eps_{i,c} ~ Uniform[-D/2, D/2], D = delta_{i,g(c)} (Figure 3 caption; the
    bound of Eq. (1)); it has zero mean and variance
    scale^2 * sum_g ||q'_{j,g}||^2 * delta_{i,g}^2 / 12.  A second-order
    Taylor expansion gives E[exp(s + delta)] ~ exp(s + Var/2), so
    b = scale^2 / 24 * sum_g n_{j,g} * delta_{i,g}^2.  Returns [Nq, Ns]."""
    n = group_sq_norms(q_rot, group)                      # [Nq, G]
    dl = np.asarray(delta, dtype=np.float64)              # [Ns, G]
    return (scale * scale / 24.0) * (n @ (dl * dl).T)


def log_sinhc(a) -> np.ndarray:
    """log(sinh(a) / a) for a >= 0, the exact log-moment of Uniform[-a, a]
    (E[exp(u)] = sinh(a)/a).

    Below a = 1 it is log1p of sinh(a)/a - 1 = sum_{k>=1} a^(2k) / (2k+1)!
    (summed to k = 12, far below fp64 resolution), which keeps full relative
    precision for small a; above, a + log((1 - exp(-2a)) / 2) - log(a)."""
    a = np.abs(np.asarray(a, dtype=np.float64))
    out = np.empty_like(a)
    small = a < 1.0
    a2 = a[small] ** 2
    term = np.ones_like(a2)
    acc = np.zeros_like(a2)
    for k in range(1, 13):
        term = term * a2 / ((2 * k) * (2 * k + 1))
        acc = acc + term
    out[small] = np.log1p(acc)
    big = ~small
    ab = a[big]
    out[big] = ab + np.log1p(-np.exp(-2.0 * ab)) - math.log(2.0) - np.log(ab)
    return out


def jensen_bias_exact(q_rot, delta, scale: float, group: int) -> np.ndarray:
    """Exact correction for independent uniform noise:
    b_ij = log E[exp(delta_ij)] = sum_c log(sinh(a_c) / a_c) with
    a_c = scale * |q'_{j,c}| * delta_{i,g(c)} / 2.  Returns [Nq, Ns].
    (The paper mentions the exact term only as the quantity the Taylor term
    approximates; this is its closed form for uniform noise.)"""
    q = np.abs(np.asarray(q_rot, dtype=np.float64))       # [Nq, d]
    dl = np.asarray(delta, dtype=np.float64)              # [Ns, G]
    nq, d = q.shape
    out = np.zeros((nq, dl.shape[0]))
    for c in range(d):
        a = 0.5 * scale * q[:, c][:, None] * dl[:, c // group][None, :]
        out += log_sinhc(a)
    return out


# ---------------------------------------------------------------------------
# Chunk attention over [cached window ; current chunk]
# ---------------------------------------------------------------------------

CORR_NONE = 0
CORR_TAYLOR = 1
CORR_EXACT = 2


def chunk_attention(q, k_hat_rot, v_hat_rot, delta_k, k_cur, v_cur, signs,
                    scale: float, group: int, corr: int = CORR_TAYLOR):
    """Attention of the current chunk's queries over the dequantized cached
    window and the unquantized current chunk, one head.

    q [Nq, d], k_cur/v_cur [Nr, d]: original basis (BF16 values as floats).
    k_hat_rot/v_hat_rot [Ns, d]: dequantized cached keys/values, rotated
    basis.  delta_k [Ns, G]: the cached keys' step sizes.

    Steps (fp64):
      q' = R q                                   (section 3, Hadamard rotation)
      cached scores  s_ij = scale * q'_j . k_hat'_i - b_ij
                     (b from ``corr``; subtracted before the softmax, cached
                     keys only: abstract, section 1)
      current scores s_ij = scale * q_j . k_i    (unquantized; (Hq)^T(Hk) = q^T k)
      p = softmax over the concatenation [cached ; current] (max-subtracted)
      P_S = sum of p over cached keys, P_R = sum over current keys
      O = sum_i p_i v_i, cached values un-rotated: v_hat = R^T v_hat'.

    Readings: no mask inside the chunk or across the window (chunk-wise
    attention); masses are per query row.  Returns (O [Nq, d], P_S [Nq],
    P_R [Nq])."""
    q = np.asarray(q, dtype=np.float64)
    kc = np.asarray(k_cur, dtype=np.float64).reshape(-1, q.shape[1])
    vc = np.asarray(v_cur, dtype=np.float64).reshape(-1, q.shape[1])
    ks = np.asarray(k_hat_rot, dtype=np.float64).reshape(-1, q.shape[1])
    vs = np.asarray(v_hat_rot, dtype=np.float64).reshape(-1, q.shape[1])
    q_rot = rotate(q, signs)
    s_cache = scale * (q_rot @ ks.T)
    if corr == CORR_TAYLOR:
        s_cache = s_cache - jensen_bias_taylor(q_rot, delta_k, scale, group)
    elif corr == CORR_EXACT:
        s_cache = s_cache - jensen_bias_exact(q_rot, delta_k, scale, group)
    elif corr != CORR_NONE:
        raise ValueError("unknown correction mode")
    s_cur = scale * (q @ kc.T)
    s = np.concatenate([s_cache, s_cur], axis=1)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    denom = e.sum(axis=1, keepdims=True)
    p = e / denom
    ns = ks.shape[0]
    p_s = p[:, :ns].sum(axis=1)
    p_r = p[:, ns:].sum(axis=1)
    v_hat = unrotate(vs, signs)
    o = p[:, :ns] @ v_hat + p[:, ns:] @ vc
    return o, p_s, p_r


# ---------------------------------------------------------------------------
# Sliding-window ring of chunk slots (host bookkeeping of the cache)
# ---------------------------------------------------------------------------


def ring_append(length: int, head_slot: int, n_new: int, chunk_tokens: int,
                n_chunks: int):
    """Where an append of ``n_new`` tokens lands and the cache state after it.

    The cache holds the last ``n_chunks`` chunks (the sliding window over the
    last n cached chunks of MAGI-1, paper section 1) in ``n_chunks`` slots of
    ``chunk_tokens`` tokens; attention reads tokens [0, length).  Rules:
      * 0 <= n_new <= chunk_tokens; n_new == 0 changes nothing;
      * while the cache is not full, every earlier slot must be full
        (length == head_slot * chunk_tokens); the chunk goes to slot
        head_slot and length grows by n_new -- so a partial chunk can only be
        the last one appended;
      * once full, only whole chunks may overwrite the oldest slot.
    Returns (first_token, new_length, new_head_slot), or None when the append
    is refused."""
    cap = chunk_tokens * n_chunks
    if n_new < 0 or n_new > chunk_tokens:
        return None
    first = head_slot * chunk_tokens
    if n_new == 0:
        return first, length, head_slot
    if length < cap:
        if length != first:
            return None
        return first, length + n_new, (head_slot + 1) % n_chunks
    if n_new != chunk_tokens:
        return None
    return first, cap, (head_slot + 1) % n_chunks
