"""GPU parity of the rotation and the quantize-append kernel against the
oracle: bit-exact (fp32 rotation values, packed codes, BF16 step sizes and
zero points), through the C-ABI."""
import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O
from quantized_kv_cache_quantize_gb300 import kvq, synth

pytestmark = pytest.mark.gpu

COMBOS = [(d, b, g) for d in (64, 128) for b in (2, 4) for g in (32, 64)]


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("d", [64, 128])
def test_rotation_fp32_bitexact(d):
    rng = np.random.default_rng(100 + d)
    x = _bf16(rng.standard_normal((1000, d)) * rng.uniform(0.01, 50, (1000, 1)))
    x[0] = 0
    s = synth.hadamard_signs(d, seed=d)
    got = kvq.rotate(x.cuda(), s, torch.float32).cpu().numpy()
    want = O.rotate_fp32(x.float().numpy(), s)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    got16 = kvq.rotate(x.cuda(), s, torch.float16).cpu().numpy()
    assert np.array_equal(got16, want.astype(np.float16))


def _expected_cache(xk, signs, bits, group, cap, first, n):
    """Oracle codes / (step, zero) of rows xk [B, H, n, d] landing at tokens
    [first, first + n)."""
    packed, delta, zero, _, _ = O.quantize_rows(xk.float().numpy(), signs, bits, group)
    return packed, O.bf16_bits(delta), O.bf16_bits(zero)


def _check_slot(cache, which, x, signs, first, n):
    packed, dbits, zbits = _expected_cache(x, signs, cache.bits, cache.group, cache.capacity,
                                           first, n)
    codes = cache.codes_view(which)[:, :, first:first + n].cpu().numpy()
    sz = cache.sz_view(which)[:, :, first:first + n].cpu().numpy().view(np.uint16)
    assert np.array_equal(codes, packed), f"{which} codes differ"
    assert np.array_equal(sz[..., 0], dbits), f"{which} step sizes differ"
    assert np.array_equal(sz[..., 1], zbits), f"{which} zero points differ"


@pytest.mark.parametrize("d,bits,group", COMBOS)
def test_append_bitexact_ring(d, bits, group):
    """Fill a 3-slot window with ragged 37-token chunks, wrap around once,
    over 2 x 3 heads; every slot matches the oracle bit for bit."""
    rng = np.random.default_rng(d * 100 + bits * 10 + group)
    B, H, C, n = 2, 3, 37, 3
    s = synth.hadamard_signs(d, seed=bits)
    cache = kvq.KVCache(B, H, d, bits, group, C, n, s)
    for step in range(n + 1):
        k = _bf16(rng.standard_normal((B, H, C, d)) * 3 + rng.standard_normal((1, 1, 1, d)))
        v = _bf16(rng.standard_normal((B, H, C, d)))
        first = cache.head_slot * C
        kvq.quantize_append(cache, k.cuda(), v.cuda())
        torch.cuda.synchronize()
        assert cache.len == min((step + 1) * C, n * C)
        assert cache.head_slot == (step + 1) % n
        _check_slot(cache, "k", k, s, first, C)
        _check_slot(cache, "v", v, s, first, C)


@pytest.mark.parametrize("d,bits,group", [(128, 2, 32), (64, 4, 64), (64, 2, 32)])
def test_append_partial_and_degenerate(d, bits, group):
    """A partial last chunk; rows with constant groups, all-zero rows,
    all-positive rows, tiny and huge magnitudes, and (d = 64) a row whose
    rotated values sit exactly on half steps: 12 e_1 rotates to +-1.5, so
    D = 1 and both the zero point and the codes are exact ties."""
    s = synth.hadamard_signs(d)
    cache = kvq.KVCache(1, 2, d, bits, group, 16, 2, np.ones(d, np.float32))
    rows = np.zeros((1, 2, 16, d), np.float32)
    rng = np.random.default_rng(7)
    rows[0, 0, 1] = 1.5                      # constant row: rotation concentrates it
    rows[0, 0, 2] = np.abs(rng.standard_normal(d)) + 4
    rows[0, 0, 3] = rng.standard_normal(d) * 1e-30
    rows[0, 0, 4] = rng.standard_normal(d) * 1e30
    rows[0, 1] = rng.standard_normal((16, d))
    rows[0, 1, 5, :group] = 0.25
    rows[0, 1, 6] = 0.0
    rows[0, 1, 6, 1] = 12.0
    k = _bf16(rows)
    v = _bf16(rows[:, ::-1].copy())
    kvq.quantize_append(cache, k.cuda(), v.cuda())
    kvq.quantize_append(cache, k[:, :, :5].contiguous().cuda(), v[:, :, :5].contiguous().cuda())
    torch.cuda.synchronize()
    assert cache.len == 21
    ones = np.ones(d, np.float32)
    _check_slot(cache, "k", k, ones, 0, 16)
    _check_slot(cache, "v", v, ones, 0, 16)
    _check_slot(cache, "k", k[:, :, :5], ones, 16, 5)
    with pytest.raises(kvq.KVQError) as e:
        kvq.quantize_append(cache, k.cuda(), v.cuda())
    assert e.value.status == kvq.KVQ_ERR_CAPACITY


@pytest.mark.parametrize("name", ["tiny", "w4_int2", "w4_int4"])
def test_append_workload_chunk(name):
    """One full chunk of the workload's key/value distribution (all heads),
    bit-exact: outlier channels, per-channel offsets."""
    w = synth.WORKLOADS[name]
    x = synth.inputs(w, n_q=1, n_s=1, n_r=1)
    s = synth.hadamard_signs(w.head_dim)
    cache = kvq.KVCache(1, w.heads, w.head_dim, w.bits, w.group, w.chunk_tokens, w.n_chunks, s)
    kvq.quantize_append(cache, x["k_new"].cuda(), x["v_new"].cuda())
    torch.cuda.synchronize()
    _check_slot(cache, "k", x["k_new"], s, 0, w.chunk_tokens)
    _check_slot(cache, "v", x["v_new"], s, 0, w.chunk_tokens)


def _check_key_channel_slot(cache, x, signs, slot, n):
    """Per-channel keys of one appended chunk x [B, H, n, d] in slot `slot`:
    packed codes per token and (step, zero) per block and channel, against
    the oracle's per-channel quantizer, bit for bit."""
    C = cache.chunk_tokens
    first = slot * C
    codes = cache.codes_view("k")[:, :, first:first + n].cpu().numpy()
    meta = cache.sz_view("k")[:, :, slot].cpu().numpy().view(np.uint16)   # [B, H, bpc, d, 2]
    nb = -(-n // kvq.KEY_BLOCK)
    for b in range(x.shape[0]):
        for h in range(x.shape[1]):
            packed, delta, zero, _, _ = O.quantize_key_chunk(x[b, h].float().numpy(), signs, cache.bits)
            assert np.array_equal(codes[b, h], packed), f"key codes differ (b{b} h{h})"
            assert np.array_equal(meta[b, h, :nb, :, 0], O.bf16_bits(delta)), "key steps differ"
            assert np.array_equal(meta[b, h, :nb, :, 1], O.bf16_bits(zero)), "key zero points differ"


@pytest.mark.parametrize("d,bits,group", [(128, 2, 32), (128, 4, 64), (64, 2, 32), (64, 4, 64)])
def test_append_key_channels_bitexact_ring(d, bits, group):
    """Per-channel key mode: 300-token chunks (two full 128-token blocks and a
    44-token one) filling a 3-slot window and wrapping once, then a partial
    chunk after a reset; keys bit-exact per block and channel, values
    bit-exact per token and group."""
    rng = np.random.default_rng(d + bits)
    B, H, C, n = 1, 3, 300, 3
    s = synth.hadamard_signs(d, seed=5)
    cache = kvq.KVCache(B, H, d, bits, group, C, n, s, key_mode=kvq.KEYS_PER_CHANNEL)
    for step in range(n + 1):
        k = rng.standard_normal((B, H, C, d)) * 2 + rng.standard_normal((1, 1, 1, d)) * 3
        k[..., :3] *= 10                                   # outlier channels
        k = _bf16(k)
        v = _bf16(rng.standard_normal((B, H, C, d)))
        slot = cache.head_slot
        kvq.quantize_append(cache, k.cuda(), v.cuda())
        torch.cuda.synchronize()
        _check_key_channel_slot(cache, k, s, slot, C)
        _check_slot(cache, "v", v, s, slot * C, C)
    part = kvq.KVCache(B, H, d, bits, group, C, n, s, key_mode=kvq.KEYS_PER_CHANNEL)
    kvq.quantize_append(part, k.cuda(), v.cuda())
    kvq.quantize_append(part, k[:, :, :1].contiguous().cuda(), v[:, :, :1].contiguous().cuda())
    torch.cuda.synchronize()
    assert part.len == C + 1
    _check_key_channel_slot(part, k[:, :, :1], s, 1, 1)
    _check_slot(part, "v", v[:, :, :1], s, C, 1)


@pytest.mark.parametrize("name", ["w4_int2", "hires_t3"])
def test_append_key_channels_workload_chunk(name):
    """One full chunk of the workload (all heads) in the per-channel key mode,
    bit-exact: 4680 or 14400 tokens, the last block partial."""
    w = synth.WORKLOADS[name]
    x = synth.inputs(w, n_q=1, n_s=1, n_r=1)
    s = synth.hadamard_signs(w.head_dim)
    cache = kvq.KVCache(1, w.heads, w.head_dim, w.bits, w.group, w.chunk_tokens, w.n_chunks, s,
                        key_mode=kvq.KEYS_PER_CHANNEL)
    kvq.quantize_append(cache, x["k_new"].cuda(), x["v_new"].cuda())
    torch.cuda.synchronize()
    _check_key_channel_slot(cache, x["k_new"], s, 0, w.chunk_tokens)
    _check_slot(cache, "v", x["v_new"], s, 0, w.chunk_tokens)
