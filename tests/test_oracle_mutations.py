"""Plant plausible mistakes in the oracle (CPU only) and check that at least
one pin catches each of them.  The mistakes are planted by monkeypatching the
oracle module for the duration of one test; nothing is changed on disk."""
import numpy as np
import pytest

from oracle import kvq_oracle as O
from tests import oracle_pins as P


def _caught():
    for check in P.ALL_CHECKS:
        try:
            check()
        except AssertionError:
            return check.__name__
    return None


def _bias_sign_flipped(q_rot, delta, scale, group):
    n = O.group_sq_norms(q_rot, group)
    return -(scale * scale / 24.0) * (n @ (np.asarray(delta, np.float64) ** 2).T)


def _bias_factor_12(q_rot, delta, scale, group):
    n = O.group_sq_norms(q_rot, group)
    return (scale * scale / 12.0) * (n @ (np.asarray(delta, np.float64) ** 2).T)


def _bias_unrotated_norms(q_rot, delta, scale, group):
    # norms of the wrong (first-group-only) slice: a dropped term
    n = O.group_sq_norms(q_rot, group)
    n[:, 1:] = 0
    return (scale * scale / 24.0) * (n @ (np.asarray(delta, np.float64) ** 2).T)


def _unrotate_transposed(y, signs):
    return np.asarray(y, dtype=np.float64) @ O.rotation_matrix(signs).T


def _rotation_wrong_norm(signs):
    s = np.asarray(signs, dtype=np.float64)
    return O.sylvester_hadamard(s.shape[0]) * s[None, :] / s.shape[0]


_real_quantize = O.quantize_groups


def _quantize_floor(y, bits, group):
    y = np.asarray(y, dtype=np.float32)
    lead, d = y.shape[:-1], y.shape[-1]
    yg = y.reshape(*lead, d // group, group)
    mn, mx = yg.min(-1), yg.max(-1)
    qmax = np.float32(2 ** bits - 1)
    delta = O.bf16_round((mx - mn) / qmax)
    delta = np.where(delta == 0, np.float32(1), delta).astype(np.float32)
    zero = O.bf16_round(np.rint(-mn / delta) + np.float32(0))
    codes = np.clip(np.floor(yg / delta[..., None]) + zero[..., None], 0, qmax)
    return codes.astype(np.uint8).reshape(*lead, d), delta, zero


def _quantize_no_zero_point(y, bits, group):
    codes, delta, zero = _real_quantize(y, bits, group)
    return codes, delta, np.zeros_like(zero)


_real_pack = O.pack_codes


def _pack_swapped_halves(codes, bits):
    c = np.asarray(codes)
    sw = c.reshape(*c.shape[:-1], -1, 2)[..., ::-1].reshape(c.shape)
    return _real_pack(sw, bits)


_real_attention = O.chunk_attention


def _attention_drops_current(q, ks, vs, dk, kc, vc, signs, scale, group, corr=O.CORR_TAYLOR):
    d = np.asarray(q).shape[1]
    z = np.zeros((0, d))
    o, ps, pr = _real_attention(q, ks, vs, dk, z, z, signs, scale, group, corr)
    return o, ps, pr + 0 * ps


def _attention_bias_on_current_too(q, ks, vs, dk, kc, vc, signs, scale, group,
                                   corr=O.CORR_TAYLOR):
    o, ps, pr = _real_attention(q, ks, vs, dk, kc, vc, signs, scale, group, corr)
    # wrong: the current chunk's values un-rotated as if they were cached
    kc = np.asarray(kc, np.float64).reshape(-1, np.asarray(q).shape[1])
    if kc.shape[0] == 0:
        return o, ps, pr
    return _real_attention(q, ks, vs, dk, O.rotate(kc, signs), vc, signs, scale, group, corr)


_real_fwht = O.rotate_fp32


def _fwht_no_scale(x, signs):
    return (_real_fwht(x, signs) * np.float32(np.sqrt(np.asarray(x).shape[-1]))).astype(np.float32)


_real_key_channels = O.quantize_key_channels


def _key_channels_per_token(y, bits, block=O.KEY_BLOCK):
    # wrong axis: one group per token (all its channels) instead of per channel
    y = np.asarray(y, dtype=np.float32)
    n, d = y.shape
    codes, dl, z = O.quantize_groups(y, bits, d)
    blocks = O.chunk_blocks(n, block)
    return (codes, np.stack([np.full(d, dl[a, 0]) for a, _ in blocks]).astype(np.float32),
            np.stack([np.full(d, z[a, 0]) for a, _ in blocks]).astype(np.float32))


def _chunk_blocks_whole_chunk(n_tokens, block=O.KEY_BLOCK):
    # wrong partition: one block over the whole chunk
    return [(0, n_tokens)]


_real_log_sinhc = O.log_sinhc


def _exact_no_half(q_rot, delta, scale, group):
    # a_c without the factor 1/2 (noise half-width taken as the whole step)
    q = np.abs(np.asarray(q_rot, dtype=np.float64))
    dl = np.asarray(delta, dtype=np.float64)
    out = np.zeros((q.shape[0], dl.shape[0]))
    for c in range(q.shape[1]):
        out += _real_log_sinhc(scale * q[:, c][:, None] * dl[:, c // group][None, :])
    return out


def _exact_group_norms(q_rot, delta, scale, group):
    # one uniform term per group with the group's query norm, instead of one
    # per channel
    n = np.sqrt(O.group_sq_norms(q_rot, group))
    dl = np.asarray(delta, dtype=np.float64)
    out = np.zeros((n.shape[0], dl.shape[0]))
    for g in range(n.shape[1]):
        out += _real_log_sinhc(0.5 * scale * n[:, g][:, None] * dl[:, g][None, :])
    return out


def _log_sinh_without_division(a):
    a = np.abs(np.asarray(a, dtype=np.float64))
    return np.log(np.sinh(np.maximum(a, 1e-300)))


def _bf16_truncate(x):
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    return (a.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).reshape(a.shape)


def _dequantize_plus_zero(codes, delta, zero, group):
    c = np.asarray(codes, dtype=np.float64)
    lead, d = c.shape[:-1], c.shape[-1]
    cg = c.reshape(*lead, d // group, group)
    out = (cg + np.asarray(zero, np.float64)[..., None]) * np.asarray(delta, np.float64)[..., None]
    return out.reshape(*lead, d)


def _rotation_signs_on_output(signs):
    # diag(signs) * H instead of H * diag(signs)
    s = np.asarray(signs, dtype=np.float64)
    return s[:, None] * O.sylvester_hadamard(s.shape[0]) / np.sqrt(s.shape[0])


_real_token_steps = O.key_channel_token_steps


def _token_steps_first_block(values, n_tokens, block=O.KEY_BLOCK):
    v = np.asarray(values)
    return np.repeat(v[:1], n_tokens, axis=0)


def _attention_masses_swapped(q, ks, vs, dk, kc, vc, signs, scale, group, corr=O.CORR_TAYLOR):
    o, ps, pr = _real_attention(q, ks, vs, dk, kc, vc, signs, scale, group, corr)
    return o, pr, ps


def _attention_exact_uses_taylor(q, ks, vs, dk, kc, vc, signs, scale, group, corr=O.CORR_TAYLOR):
    if corr == O.CORR_EXACT:
        corr = O.CORR_TAYLOR
    return _real_attention(q, ks, vs, dk, kc, vc, signs, scale, group, corr)


_real_ring = O.ring_append


def _ring_no_wrap(length, head_slot, n_new, chunk_tokens, n_chunks):
    r = _real_ring(length, head_slot, n_new, chunk_tokens, n_chunks)
    if r is None:
        return None
    start, new_len, nxt = r
    return start, new_len, min(head_slot + 1, n_chunks - 1)


def _rotation_bounds_no_error(x, signs):
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[-1]
    w = O.sylvester_hadamard(d) * np.asarray(signs, np.float64)[None, :]
    inv = np.float64(np.float32(1.0 / np.sqrt(d)))
    y = ((x.astype(np.float64) @ w.T).astype(np.float32).astype(np.float64) * inv).astype(np.float32)
    return y, y


_real_admissible = O.quantize_groups_admissible


def _admissible_zero_one_end(y_lo, y_hi, bits, group):
    cd, cz, clo, chi = _real_admissible(y_lo, y_hi, bits, group)
    cz = cz.copy()
    cz[..., 1] = cz[..., 0]
    cz[..., 3] = cz[..., 2]
    return cd, cz, clo, chi


def _admissible_codes_any(y_lo, y_hi, bits, group):
    cd, cz, clo, chi = _real_admissible(y_lo, y_hi, bits, group)
    return cd, cz, np.zeros_like(clo), np.full_like(chi, 2 ** bits - 1)


def _key_admissible_along_channels(y_lo, y_hi, bits, block=O.KEY_BLOCK):
    # a full block grouped along channels (per token) instead of along
    # tokens: the transpose forgotten (shapes agree when the block has d tokens)
    lo = np.asarray(y_lo, np.float32)
    hi = np.asarray(y_hi, np.float32)
    out = []
    for a, b in O.chunk_blocks(lo.shape[0], block):
        n = b - a
        if n == lo.shape[1]:
            cd, cz, clo, chi = _real_admissible(lo[a:b], hi[a:b], bits, n)
        else:
            cd, cz, clo, chi = _real_admissible(np.ascontiguousarray(lo[a:b].T),
                                                np.ascontiguousarray(hi[a:b].T), bits, n)
        out.append((cd[:, 0], cz[:, 0], clo[:, 0], chi[:, 0]))
    return out


MUTANTS = {
    "key_admissible_along_channels": ("quantize_key_channels_admissible", _key_admissible_along_channels),
    "rotation_bounds_no_error": ("rotation_bounds", _rotation_bounds_no_error),
    "admissible_zero_one_end": ("quantize_groups_admissible", _admissible_zero_one_end),
    "admissible_codes_any": ("quantize_groups_admissible", _admissible_codes_any),
    "key_channels_per_token": ("quantize_key_channels", _key_channels_per_token),
    "key_blocks_whole_chunk": ("chunk_blocks", _chunk_blocks_whole_chunk),
    "bias_sign_flipped": ("jensen_bias_taylor", _bias_sign_flipped),
    "bias_factor_12": ("jensen_bias_taylor", _bias_factor_12),
    "bias_dropped_group_terms": ("jensen_bias_taylor", _bias_unrotated_norms),
    "unrotate_transposed": ("unrotate", _unrotate_transposed),
    "rotation_wrong_norm": ("rotation_matrix", _rotation_wrong_norm),
    "quantize_floor": ("quantize_groups", _quantize_floor),
    "quantize_no_zero_point": ("quantize_groups", _quantize_no_zero_point),
    "pack_swapped_pairs": ("pack_codes", _pack_swapped_halves),
    "attention_drops_current": ("chunk_attention", _attention_drops_current),
    "attention_rotates_current_keys": ("chunk_attention", _attention_bias_on_current_too),
    "fwht_no_scale": ("rotate_fp32", _fwht_no_scale),
    "exact_no_half": ("jensen_bias_exact", _exact_no_half),
    "exact_group_norms": ("jensen_bias_exact", _exact_group_norms),
    "log_sinh_without_division": ("log_sinhc", _log_sinh_without_division),
    "bf16_truncate": ("bf16_round", _bf16_truncate),
    "dequantize_plus_zero": ("dequantize", _dequantize_plus_zero),
    "rotation_signs_on_output": ("rotation_matrix", _rotation_signs_on_output),
    "key_steps_first_block": ("key_channel_token_steps", _token_steps_first_block),
    "attention_masses_swapped": ("chunk_attention", _attention_masses_swapped),
    "attention_exact_uses_taylor": ("chunk_attention", _attention_exact_uses_taylor),
    "ring_no_wrap": ("ring_append", _ring_no_wrap),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    assert _caught() is not None, f"no pin caught the planted mistake {name}"
