"""GPU parity of the rotation and the quantize-append kernel against the
oracle, through the C-ABI.

The per-token quantizer rotates on the tensor cores: every product of a
BF16 value with a +-1 entry is exact, but the hardware chooses the fp32
summation order.  So its fp32 rotation is checked to lie inside the oracle's
bounds for any fp32 summation (O.rotation_bounds), and to equal the
butterfly result bit for bit on rows whose partial sums are all fp32
numbers; and its codes, step sizes and zero points are checked to be one of
the answers Eq. (1) gives inside those bounds (O.quantize_groups_admissible):
the same answer, bit for bit, wherever the bounds fix it, which is almost
everywhere and everywhere on such rows.  The FP16 rotation (the attention's
operands) and the per-channel key quantizer keep the butterfly order and are
bit-exact against O.rotate_fp32."""
import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O
from quantized_kv_cache_quantize_gb300 import kvq, synth
from tests.gpu_common import admissible

pytestmark = pytest.mark.gpu

COMBOS = [(d, b, g) for d in (64, 128) for b in (2, 4) for g in (32, 64)]


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)


def _grid(rng, shape, scale_exp=12):
    """BF16 rows m * 2^e (|m| <= 255, one e per row): every partial sum of a
    row's rotation is an fp32 number, so any summation order is exact."""
    m = np.clip(np.rint(rng.standard_normal(shape) * 40), -255, 255)
    e = rng.integers(-scale_exp, scale_exp, shape[:-1] + (1,)).astype(np.float64)
    return _bf16(m * 2.0 ** e)


@pytest.mark.parametrize("d", [64, 128])
def test_rotation_fp16_bitexact(d):
    """The attention's FP16 operands: the butterfly order, bit for bit."""
    rng = np.random.default_rng(100 + d)
    x = _bf16(rng.standard_normal((1000, d)) * rng.uniform(0.01, 50, (1000, 1)))
    x[0] = 0
    s = synth.hadamard_signs(d, seed=d)
    got16 = kvq.rotate(x.cuda(), s, torch.float16).cpu().numpy()
    assert np.array_equal(got16, O.rotate_fp32(x.float().numpy(), s).astype(np.float16))


@pytest.mark.parametrize("d", [64, 128])
def test_rotation_fp32_bounds(d):
    """The quantizer's fp32 rotation (kvq_rotate's fp32 output): inside the
    oracle's bounds for any summation order; exact on grid rows; the same
    bits for a row wherever it sits in the input (tiles of 128 rows, ragged
    last tile)."""
    rng = np.random.default_rng(200 + d)
    x = _bf16(rng.standard_normal((1000, d)) * rng.uniform(0.01, 50, (1000, 1)))
    x[:, :3] *= 12
    x[0] = 0
    s = synth.hadamard_signs(d, seed=d)
    got = kvq.rotate(x.cuda(), s, torch.float32).cpu().numpy()
    lo, hi = O.rotation_bounds(x.float().numpy(), s)
    assert np.all((lo <= got) & (got <= hi))
    xg = _grid(rng, (333, d))
    gotg = kvq.rotate(xg.cuda(), s, torch.float32).cpu().numpy()
    # (values: a zero may carry either sign)
    assert np.array_equal(gotg, O.rotate_fp32(xg.float().numpy(), s))
    perm = np.roll(np.arange(1000), 357)
    got2 = kvq.rotate(x[perm].contiguous().cuda(), s, torch.float32).cpu().numpy()
    assert np.array_equal(got2, got[perm])


def _check_slot(cache, which, x, signs, first, n, min_unique=0.99):
    """The slot's codes and (step, zero) records of rows x [B, H, n, d]
    against the oracle's admissible answers; `min_unique` of the codes must
    be fixed by the bounds (1.0 on grid rows)."""
    codes = cache.codes_view(which)[:, :, first:first + n].cpu().numpy()
    sz = cache.sz_view(which)[:, :, first:first + n].cpu().numpy()
    ok, unique = admissible(x, signs, cache.bits, cache.group, codes, sz)
    assert ok.all(), f"{which}: {int((~ok).sum())} groups outside the admissible answers"
    assert unique >= min_unique, f"{which}: only {unique:.5f} of the codes determined"
    # zero points are stored as +0, never -0
    assert not np.any(sz.view(np.uint16)[..., 1] == 0x8000)


@pytest.mark.parametrize("d,bits,group", COMBOS)
def test_append_ring(d, bits, group):
    """Fill a 3-slot window with ragged 37-token chunks, wrap around once,
    over 2 x 3 heads; every slot holds an admissible answer, and on the
    steps with grid rows (exact sums) exactly the oracle's one answer."""
    rng = np.random.default_rng(d * 100 + bits * 10 + group)
    B, H, C, n = 2, 3, 37, 3
    s = synth.hadamard_signs(d, seed=bits)
    cache = kvq.KVCache(B, H, d, bits, group, C, n, s)
    for step in range(n + 1):
        grid = step % 2 == 1
        if grid:
            k, v = _grid(rng, (B, H, C, d)), _grid(rng, (B, H, C, d))
        else:
            k = _bf16(rng.standard_normal((B, H, C, d)) * 3 + rng.standard_normal((1, 1, 1, d)))
            v = _bf16(rng.standard_normal((B, H, C, d)))
        first = cache.head_slot * C
        kvq.quantize_append(cache, k.cuda(), v.cuda())
        torch.cuda.synchronize()
        assert cache.len == min((step + 1) * C, n * C)
        assert cache.head_slot == (step + 1) % n
        _check_slot(cache, "k", k, s, first, C, 1.0 if grid else 0.99)
        _check_slot(cache, "v", v, s, first, C, 1.0 if grid else 0.99)
        if grid:
            packed, delta, zero, _, _ = O.quantize_rows(k.float().numpy(), s, bits, group)
            assert np.array_equal(cache.codes_view("k")[:, :, first:first + C].cpu().numpy(), packed)


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


@pytest.mark.parametrize("name", ["tiny", "w4_int2", "w4_int4", "w8_int2", "hires_t3"])
def test_append_workload_chunk(name):
    """One full chunk of the workload's key/value distribution (all heads):
    outlier channels, per-channel offsets; admissible answers, and the
    bounds fix at least 99 % of the codes."""
    w = synth.WORKLOADS[name]
    x = synth.inputs(w, n_q=1, n_s=1, n_r=1)
    s = synth.hadamard_signs(w.head_dim)
    cache = kvq.KVCache(1, w.heads, w.head_dim, w.bits, w.group, w.chunk_tokens, w.n_chunks, s)
    kvq.quantize_append(cache, x["k_new"].cuda(), x["v_new"].cuda())
    torch.cuda.synchronize()
    _check_slot(cache, "k", x["k_new"], s, 0, w.chunk_tokens)
    _check_slot(cache, "v", x["v_new"], s, 0, w.chunk_tokens)


def _check_key_channel_slot(cache, x, signs, slot, n, min_unique=0.99):
    """Per-channel keys of one appended chunk x [B, H, n, d] in slot `slot`:
    packed codes per token and (step, zero) per block and channel, against
    the oracle's admissible answers for the rotation known to within its
    fp32 summation bound; `min_unique` of the codes must be fixed by the
    bounds (1.0 on grid rows, which the oracle then matches bit for bit)."""
    C = cache.chunk_tokens
    first = slot * C
    d = cache.head_dim
    codes = cache.codes_view("k")[:, :, first:first + n].cpu().numpy()
    meta = cache.sz_view("k")[:, :, slot].cpu().numpy().view(np.uint16)   # [B, H, bpc, d, 2]
    fixed = total = 0
    for b in range(x.shape[0]):
        for h in range(x.shape[1]):
            lo, hi = O.rotation_bounds(x[b, h].float().numpy(), signs)
            got = O.unpack_codes(codes[b, h], cache.bits, d)                  # [n, d]
            for i, ((a0, a1), (cd, cz, clo, chi)) in enumerate(
                    zip(O.chunk_blocks(n), O.quantize_key_channels_admissible(lo, hi, cache.bits))):
                g = got[a0:a1].T[:, None, :]                                  # [d, 1, tokens]
                ok = ((O.bf16_bits(cd) == meta[b, h, i, :, 0][:, None]) &
                      (O.bf16_bits(cz) == meta[b, h, i, :, 1][:, None]) &
                      np.all((clo <= g) & (g <= chi), axis=-1))
                assert ok.any(axis=-1).all(), f"key block {i} (b{b} h{h}) outside the admissible answers"
                fixed += int(np.sum(clo == chi))
                total += clo.size
    assert fixed / total >= min_unique, f"only {fixed / total:.5f} of the key codes determined"


@pytest.mark.parametrize("d,bits,group", [(128, 2, 32), (128, 4, 64), (64, 2, 32), (64, 4, 64)])
def test_append_key_channels_bitexact_ring(d, bits, group):
    """Per-channel key mode: 300-token chunks (two full 128-token blocks and a
    44-token one) filling a 3-slot window and wrapping once, then a partial
    chunk after a reset; keys per block and channel and values per token and
    group among the oracle's admissible answers (grid rows on the last step:
    exactly the oracle's answer)."""
    rng = np.random.default_rng(d + bits)
    B, H, C, n = 1, 3, 300, 3
    s = synth.hadamard_signs(d, seed=5)
    cache = kvq.KVCache(B, H, d, bits, group, C, n, s, key_mode=kvq.KEYS_PER_CHANNEL)
    for step in range(n + 1):
        grid = step == n
        if grid:
            k = _grid(rng, (B, H, C, d))
        else:
            k = rng.standard_normal((B, H, C, d)) * 2 + rng.standard_normal((1, 1, 1, d)) * 3
            k[..., :3] *= 10                                   # outlier channels
            k = _bf16(k)
        v = _bf16(rng.standard_normal((B, H, C, d)))
        slot = cache.head_slot
        kvq.quantize_append(cache, k.cuda(), v.cuda())
        torch.cuda.synchronize()
        _check_key_channel_slot(cache, k, s, slot, C, 1.0 if grid else 0.99)
        _check_slot(cache, "v", v, s, slot * C, C)
        if grid:
            packed = O.quantize_key_chunk(k[0, 0].float().numpy(), s, bits)[0]
            assert np.array_equal(cache.codes_view("k")[0, 0, slot * C:(slot + 1) * C].cpu().numpy(), packed)
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
    keys and values among the admissible answers: 4680 or 14400 tokens, the
    last block partial."""
    w = synth.WORKLOADS[name]
    x = synth.inputs(w, n_q=1, n_s=1, n_r=1)
    s = synth.hadamard_signs(w.head_dim)
    cache = kvq.KVCache(1, w.heads, w.head_dim, w.bits, w.group, w.chunk_tokens, w.n_chunks, s,
                        key_mode=kvq.KEYS_PER_CHANNEL)
    kvq.quantize_append(cache, x["k_new"].cuda(), x["v_new"].cuda())
    torch.cuda.synchronize()
    _check_key_channel_slot(cache, x["k_new"], s, 0, w.chunk_tokens)
    _check_slot(cache, "v", x["v_new"], s, 0, w.chunk_tokens)


def test_append_waits_for_the_previous_attention():
    """The append is launched so that its start may overlap the end of the
    kernel before it in the stream; it must not write the cache slot that
    kernel still reads.  A full window, an attention call over it and, with
    no synchronization between them, an append overwriting the oldest slot:
    the attention's output is the one computed before the append, bit for
    bit (the attention kernels are deterministic)."""
    w = synth.WORKLOADS["w4_int2"]
    x = synth.inputs(w, n_q=512, n_r=256)
    s = synth.hadamard_signs(w.head_dim)
    cache = kvq.KVCache(1, w.heads, w.head_dim, w.bits, w.group, w.chunk_tokens, w.n_chunks, s)
    kw, vw = x["k_win"].cuda(), x["v_win"].cuda()
    for c in range(w.n_chunks):
        sl = slice(c * w.chunk_tokens, (c + 1) * w.chunk_tokens)
        kvq.quantize_append(cache, kw[:, :, sl].contiguous(), vw[:, :, sl].contiguous())
    q, kc, vc = x["q"].cuda(), x["k_cur"].cuda(), x["v_cur"].cuda()
    ref = kvq.attention_corrected(cache, q, kc, vc)
    torch.cuda.synchronize()
    kn, vn = x["k_new"].cuda(), x["v_new"].cuda()
    for _ in range(3):
        out = kvq.attention_corrected(cache, q, kc, vc)
        kvq.quantize_append(cache, kn, vn)          # overwrites a slot the attention reads
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        # put the window back: the same chunks in the same slots
        c = (cache.head_slot - 1) % w.n_chunks
        sl = slice(c * w.chunk_tokens, (c + 1) * w.chunk_tokens)
        cache.struct.head_slot = c
        kvq.quantize_append(cache, kw[:, :, sl].contiguous(), vw[:, :, sl].contiguous())
    assert kvq.last_device_status() == kvq.KVQ_OK


@pytest.mark.parametrize("d,bits,group", [(128, 2, 32), (128, 4, 64), (64, 2, 32)])
def test_append_division_route(d, bits, group):
    """Rows scaled near 2^-112 (grid values m 2^e, |m| <= 255, so the sums are
    exact): every step is below 2^-100, where Eq. (1)'s quotients leave the
    reciprocal route for one IEEE division per value -- per token and group
    (keys and values) and, in the per-channel key mode, per channel; the
    oracle's answer bit for bit."""
    rng = np.random.default_rng(900 + d + bits)
    B, H, C = 1, 2, 200
    s = synth.hadamard_signs(d, seed=9)
    m = np.clip(np.rint(rng.standard_normal((B, H, C, d)) * 40), -255, 255)
    k = _bf16(m * 2.0 ** rng.integers(-114, -110, (B, H, C, 1)).astype(np.float64))
    m = np.clip(np.rint(rng.standard_normal((B, H, C, d)) * 40), -255, 255)
    v = _bf16(m * 2.0 ** rng.integers(-114, -110, (B, H, C, 1)).astype(np.float64))
    assert float(k.abs().max()) < 2.0 ** -100
    cache = kvq.KVCache(B, H, d, bits, group, C, 2, s)
    kvq.quantize_append(cache, k.cuda(), v.cuda())
    torch.cuda.synchronize()
    for which, x in (("k", k), ("v", v)):
        packed, delta, zero, _, _ = O.quantize_rows(x.float().numpy(), s, bits, group)
        assert float(np.max(delta)) < 2.0 ** -100
        assert np.array_equal(cache.codes_view(which)[:, :, :C].cpu().numpy(), packed), which
        sz = cache.sz_view(which)[:, :, :C].cpu().numpy().view(np.uint16)
        assert np.array_equal(sz[..., 0], O.bf16_bits(delta)) and np.array_equal(sz[..., 1], O.bf16_bits(zero))
    kc = kvq.KVCache(B, H, d, bits, group, C, 2, s, key_mode=kvq.KEYS_PER_CHANNEL)
    kvq.quantize_append(kc, k.cuda(), v.cuda())
    torch.cuda.synchronize()
    _check_key_channel_slot(kc, k, s, 0, C, 1.0)
    for h in range(H):
        packed = O.quantize_key_chunk(k[0, h].float().numpy(), s, bits)[0]
        assert np.array_equal(kc.codes_view("k")[0, h, :C].cpu().numpy(), packed)
    assert kvq.last_device_status() == kvq.KVQ_OK
