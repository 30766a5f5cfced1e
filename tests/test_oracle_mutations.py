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


MUTANTS = {
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
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    assert _caught() is not None, f"no pin caught the planted mistake {name}"
