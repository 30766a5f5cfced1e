"""Checks that pin the CPU oracle to facts outside itself.

Each ``check_*`` raises AssertionError when the oracle disagrees with what
the paper ("Quantized Keys Steal Attention: Bias Correction for KV-Cache
Compression in Video Diffusion") or plain mathematics fixes.  They are run
by ``test_oracle_pins.py`` and, with mistakes planted in the oracle, by
``test_oracle_mutations.py`` (which expects them to fail).
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

from oracle import kvq_oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            out.append(line)
    return out


# --------------------------------------------------------------------------
# Rotation (section 3, "Hadamard rotation")
# --------------------------------------------------------------------------


def check_hadamard_hand_d4():
    rows = dict(r.split(":", 1) for r in _rows("hadamard_d4.txt"))
    syl = np.array([[float(v) for v in rows[f"sylvester_row{i}"].split()] for i in range(4)])
    assert np.array_equal(O.sylvester_hadamard(4), syl)
    signs = np.array([float(v) for v in rows["signs"].split()])
    x = np.array([float(v) for v in rows["x"].split()])
    want = np.array([float(v) for v in rows["rotated"].split()])
    assert np.allclose(O.rotate(x[None], signs)[0], want, rtol=0, atol=1e-14)
    got32 = O.rotate_fp32(x[None].astype(np.float32), signs.astype(np.float32))[0]
    assert np.array_equal(got32, want.astype(np.float32))
    assert np.allclose(O.unrotate(want[None], signs)[0], x, rtol=0, atol=1e-14)


def check_rotation_orthogonal_and_score_invariant():
    rng = np.random.default_rng(1)
    for d in (2, 4, 64, 128):
        s = np.where(rng.integers(0, 2, d) == 1, -1.0, 1.0)
        r = O.rotation_matrix(s)
        assert np.abs(r @ r.T - np.eye(d)).max() < 1e-12
        q = rng.standard_normal((5, d))
        k = rng.standard_normal((7, d))
        # (Hq)^T (Hk) = q^T k
        assert np.abs(O.rotate(q, s) @ O.rotate(k, s).T - q @ k.T).max() < 1e-11
        assert np.abs(O.unrotate(O.rotate(q, s), s) - q).max() < 1e-12


def check_fwht_fp32_matches_fp64():
    rng = np.random.default_rng(2)
    for d in (64, 128):
        s = np.where(rng.integers(0, 2, d) == 1, -1.0, 1.0).astype(np.float32)
        x = (rng.standard_normal((200, d)) * 3).astype(np.float32)
        y32 = O.rotate_fp32(x, s).astype(np.float64)
        y64 = O.rotate(x.astype(np.float64), s)
        # log2(d) rounded additions + one rounded scaling per element
        bound = (math.log2(d) + 2) * 2.0 ** -24 * np.abs(x).sum(axis=1, keepdims=True) / math.sqrt(d)
        assert np.all(np.abs(y32 - y64) <= bound)
        # a basis vector e_i becomes +-fl(1/sqrt(d)) times column i of Sylvester
        e = np.eye(d, dtype=np.float32)
        inv = np.float32(1.0 / math.sqrt(d))
        want = (O.sylvester_hadamard(d).T * s[:, None]).astype(np.float32) * inv
        assert np.array_equal(O.rotate_fp32(e, s), want.astype(np.float32))


def _bf16_rows(rng, n, d):
    x = rng.standard_normal((n, d)) * rng.uniform(0.01, 50, (n, 1))
    x[:, :3] *= 12                                   # outlier channels
    return O.bf16_round(x.astype(np.float32))


def check_rotation_bounds():
    """rotation_bounds holds every fp32 summation order: the butterfly
    order, sequential sums in random orders and the exact sum (times the
    fp32 constant) all lie inside; rows on a coarse grid have exact sums, so
    their bounds collapse onto the butterfly result; the bounds are no wider
    than the recursive-summation bound allows."""
    rng = np.random.default_rng(21)
    for d in (64, 128):
        s = np.where(rng.integers(0, 2, d) == 1, -1.0, 1.0).astype(np.float32)
        x = _bf16_rows(rng, 300, d)
        lo, hi = O.rotation_bounds(x, s)
        assert lo.dtype == np.float32 and np.all(lo <= hi)
        y32 = O.rotate_fp32(x, s)
        assert np.all((lo <= y32) & (y32 <= hi))
        inv = np.float64(np.float32(1.0 / math.sqrt(d)))
        w = O.sylvester_hadamard(d) * s.astype(np.float64)[None, :]
        center = (x.astype(np.float64) @ w.T) * inv
        # the exact sum rounded to fp32 once, times the constant: one order
        c32 = ((x.astype(np.float64) @ w.T).astype(np.float32).astype(np.float64) * inv).astype(np.float32)
        assert np.all((lo <= c32) & (c32 <= hi))
        for r in range(0, 300, 15):
            for n in rng.integers(0, d, 4):
                terms = (x[r].astype(np.float64) * w[n]).astype(np.float32)   # exact products
                acc = np.float32(0.0)
                for k in rng.permutation(d):
                    acc = np.float32(acc + terms[k])
                y = np.float32(np.float64(acc) * inv)
                assert lo[r, n] <= y <= hi[r, n], (d, r, n)
        gamma = (d - 1) * 2.0 ** -23 / (1 - (d - 1) * 2.0 ** -23)
        width = (hi.astype(np.float64) - lo) / inv
        allowed = 2 * (gamma + d * 2.0 ** -53) * np.abs(x.astype(np.float64)).sum(1, keepdims=True)
        assert np.all(width <= allowed + 4 * np.spacing(np.abs(center).astype(np.float32)) / inv)
        # values m * 2^e, |m| <= 255: every partial sum is an fp32 number
        m = np.clip(np.rint(rng.standard_normal((200, d)) * 40), -255, 255)
        xg = (m * 2.0 ** rng.integers(-12, 12, (200, 1))).astype(np.float32)
        lo, hi = O.rotation_bounds(xg, s)
        assert np.array_equal(lo, hi) and np.array_equal(lo, O.rotate_fp32(xg, s))


def check_quantize_admissible():
    """quantize_groups_admissible: with exact inputs its four candidates are
    quantize_groups' one answer; with interval inputs every fp32 row inside
    the bounds (sampled: each element at its low end, its high end or a value
    between) has its quantize_groups answer among the candidates; and the
    candidate set stays tight (almost every code determined)."""
    rng = np.random.default_rng(22)
    for bits, group in ((2, 32), (4, 64), (2, 64), (4, 32)):
        y = (rng.standard_normal((400, 128)) * rng.uniform(0.1, 5, (400, 1))).astype(np.float32)
        codes, delta, zero = O.quantize_groups(y, bits, group)
        cd, cz, clo, chi = O.quantize_groups_admissible(y, y, bits, group)
        g_n = 128 // group
        cg = codes.reshape(400, g_n, group)
        for i in range(4):
            assert np.array_equal(cd[..., i], delta) and np.array_equal(cz[..., i], zero)
            assert np.array_equal(clo[..., i, :], cg) and np.array_equal(chi[..., i, :], cg)
        # bounds a few units wide around y
        ulps = rng.integers(0, 40, y.shape)
        lo = y - (np.spacing(np.abs(y)) * ulps).astype(np.float32)
        hi = y + (np.spacing(np.abs(y)) * rng.integers(0, 40, y.shape)).astype(np.float32)
        cd, cz, clo, chi = O.quantize_groups_admissible(lo, hi, bits, group)
        for _ in range(12):
            pick = rng.integers(0, 3, y.shape)
            mid = (lo + (hi - lo) * rng.uniform(0, 1, y.shape).astype(np.float32)).astype(np.float32)
            mid = np.clip(mid, lo, hi)
            ys = np.where(pick == 0, lo, np.where(pick == 1, hi, mid)).astype(np.float32)
            c, dl, z = O.quantize_groups(ys, bits, group)
            cgs = c.reshape(400, g_n, group)
            ok = ((cd == dl[..., None]) & (cz == z[..., None]) &
                  np.all((clo <= cgs[..., None, :]) & (cgs[..., None, :] <= chi), axis=-1))
            assert ok.any(axis=-1).all(), (bits, group)
        assert np.mean(clo == chi) > 0.99
    # a zero point on a tie: min -1.5, max 1.5, INT2 -> step 1 and
    # -min / step = 1.5 (rint -> 2); one unit either side of the min moves
    # the zero point to 1 or keeps it at 2, with the step unchanged
    y = np.linspace(-1.5, 1.5, 32, dtype=np.float32)[None]
    lo, hi = y.copy(), y.copy()
    lo[0, 0] = np.nextafter(np.float32(-1.5), np.float32(-2))
    hi[0, 0] = np.nextafter(np.float32(-1.5), np.float32(0))
    cd, cz, clo, chi = O.quantize_groups_admissible(lo, hi, 2, 32)
    for ys in (lo, hi, y):
        c, dl, z = O.quantize_groups(ys, 2, 32)
        ok = ((cd == dl[..., None]) & (cz == z[..., None]) &
              np.all((clo <= c[:, None, None, :]) & (c[:, None, None, :] <= chi), axis=-1))
        assert ok.any(), (ys[0, 0], z)
    assert set(np.unique(cz)) == {1.0, 2.0}


def check_key_channels_admissible():
    """quantize_key_channels_admissible: exact bounds give the per-channel
    quantizer's one answer (every block, the last one short); keys sampled
    inside interval bounds always have their answer among the candidates."""
    rng = np.random.default_rng(23)
    for d, bits in ((64, 2), (64, 4), (128, 2)):
        y = (rng.standard_normal((300, d)) * 2 + rng.standard_normal((1, d)) * 3).astype(np.float32)
        codes, delta, zero = O.quantize_key_channels(y, bits)
        blocks = O.chunk_blocks(300)
        adm = O.quantize_key_channels_admissible(y, y, bits)
        assert len(adm) == len(blocks) == 3
        for (a, b), (cd, cz, clo, chi), dl, z in zip(blocks, adm, delta, zero):
            for i in range(4):
                assert np.array_equal(cd[:, i], dl) and np.array_equal(cz[:, i], z)
                assert np.array_equal(clo[:, i, :], codes[a:b].T) and np.array_equal(chi[:, i, :], codes[a:b].T)
        lo = y - (np.spacing(np.abs(y)) * rng.integers(0, 40, y.shape)).astype(np.float32)
        hi = y + (np.spacing(np.abs(y)) * rng.integers(0, 40, y.shape)).astype(np.float32)
        # a one-token block: every channel a constant group (step |value|)
        c1, d1, z1 = O.quantize_key_channels(y[:1], bits)
        (cd1, cz1, clo1, chi1), = O.quantize_key_channels_admissible(lo[:1], hi[:1], bits)
        ok1 = ((cd1 == d1[0][:, None]) & (cz1 == z1[0][:, None]) &
               np.all((clo1 <= c1.T[:, None, :]) & (c1.T[:, None, :] <= chi1), axis=-1))
        assert ok1.any(axis=-1).all()
        (cd1, _, _, _), = O.quantize_key_channels_admissible(y[:1], y[:1], bits)
        assert np.array_equal(cd1[:, 0], d1[0]) and np.array_equal(d1[0], O.bf16_round(np.abs(y[0])))
        adm = O.quantize_key_channels_admissible(lo, hi, bits)
        for _ in range(8):
            ys = np.where(rng.integers(0, 2, y.shape) == 1, lo, hi).astype(np.float32)
            c, dl, z = O.quantize_key_channels(ys, bits)
            for (a, b), (cd, cz, clo, chi), dlb, zb in zip(blocks, adm, dl, z):
                cb = c[a:b].T[:, None, :]
                ok = ((cd == dlb[:, None]) & (cz == zb[:, None]) &
                      np.all((clo <= cb) & (cb <= chi), axis=-1))
                assert ok.any(axis=-1).all(), bits


def check_bf16_round_matches_torch():
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * 10,
        np.array([0.0, -0.0, 1.0, 1.00390625, 1.005859375, 1.0 + 2 ** -8,
                  1.0 + 3 * 2 ** -9, 65280.0, 1e-40, -3.0e38], dtype=np.float32),
    ]).astype(np.float32)
    # exact ties at both parities of the kept last bit
    ties = (np.arange(1000, dtype=np.uint32) << np.uint32(16)) | np.uint32(0x3F808000)
    x = np.concatenate([x, ties.view(np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(O.bf16_round(x), want)


# --------------------------------------------------------------------------
# Quantization (section 3, Eq. (1) and "Quantization granularity")
# --------------------------------------------------------------------------


def check_quant_hand_fixture():
    for line in _rows("quant_eq1.txt"):
        parts = [p.strip() for p in line.split("|")]
        bits = int(parts[0])
        x = np.array([float(v) for v in parts[1].split()], dtype=np.float32)
        d_want = float(parts[2])
        z_want = float(parts[3])
        c_want = np.array([int(v) for v in parts[4].split()])
        xh_want = np.array([float(v) for v in parts[5].split()])
        codes, delta, zero = O.quantize_groups(x[None], bits, x.size)
        assert float(delta[0, 0]) == d_want, (line, delta)
        assert float(zero[0, 0]) == z_want, (line, zero)
        assert np.array_equal(codes[0], c_want), (line, codes)
        xh = O.dequantize(codes, delta, zero, x.size)[0]
        assert np.array_equal(xh, xh_want), (line, xh)
        # a zero point of -0 would differ in its bits from +0
        assert O.bf16_bits(zero)[0, 0] != 0x8000


def check_quant_bounds_and_brute_force():
    """|x_hat - x| <= D/2 for elements whose code is not clamped; every code
    is the nearest grid point (brute force over all 2^B codes)."""
    rng = np.random.default_rng(4)
    for bits, group in ((2, 32), (4, 64), (2, 4), (4, 8)):
        y = (rng.standard_normal((300, 128)) * rng.uniform(0.1, 5, (300, 1))
             + rng.standard_normal((300, 1))).astype(np.float32)
        codes, delta, zero = O.quantize_groups(y, bits, group)
        qmax = 2 ** bits - 1
        assert codes.max() <= qmax
        xh = O.dequantize(codes, delta, zero, group)
        g_n = 128 // group
        dfull = np.repeat(delta, group, axis=1).astype(np.float64)
        zfull = np.repeat(zero, group, axis=1).astype(np.float64)
        err = np.abs(xh - y)
        unclamped = (codes > 0) & (codes < qmax)
        assert np.all(err[unclamped] <= dfull[unclamped] / 2 * (1 + 1e-6))
        cands = (np.arange(qmax + 1)[None, None, :] - zfull[..., None]) * dfull[..., None]
        best = np.abs(cands - y[..., None].astype(np.float64)).min(axis=-1)
        assert np.all(err <= best + 1e-6 * dfull)
        # the grid covers [min, max] up to the BF16 rounding of D
        yg = y.reshape(300, g_n, group)
        # (slack: half a step, plus qmax times the BF16 rounding of the step)
        lo = (0 - zero.astype(np.float64)) * delta
        hi = (qmax - zero.astype(np.float64)) * delta
        d_exact = (yg.max(-1).astype(np.float64) - yg.min(-1)) / qmax
        slack = delta * 0.5 + qmax * np.abs(delta - d_exact) + 1e-6 * delta
        assert np.all(lo <= yg.min(-1) + slack)
        assert np.all(hi >= yg.max(-1) - slack)
        assert np.all(np.abs(delta - (yg.max(-1) - yg.min(-1)) / qmax) <= delta * 2 ** -8 + 1e-30)


def check_smaller_groups_smaller_error():
    """Section 3 "Quantization granularity": smaller groups give a smaller
    quantization error (and more memory)."""
    rng = np.random.default_rng(5)
    y = rng.standard_normal((2000, 128)).astype(np.float32)
    y[:, :3] *= 10
    errs = []
    for g in (16, 32, 64, 128):
        c, dl, z = O.quantize_groups(y, 2, g)
        errs.append(np.abs(O.dequantize(c, dl, z, g) - y).mean())
    assert errs[0] < errs[1] < errs[2] < errs[3], errs


def check_pack_hand_fixture():
    for line in _rows("pack_layout.txt"):
        bits_s, codes_s, bytes_s = [p.strip() for p in line.split("|")]
        bits = int(bits_s)
        codes = np.array([int(v) for v in codes_s.split()], dtype=np.uint8)
        want = np.array([int(v, 16) for v in bytes_s.split()], dtype=np.uint8)
        got = O.pack_codes(codes[None], bits)[0]
        assert np.array_equal(got, want), (bits, got, want)
        assert np.array_equal(O.unpack_codes(got[None], bits, codes.size)[0], codes)


def check_pack_roundtrip():
    rng = np.random.default_rng(6)
    for bits in (2, 4):
        for d in (64, 128):
            c = rng.integers(0, 2 ** bits, (50, d)).astype(np.uint8)
            p = O.pack_codes(c, bits)
            assert p.shape == (50, d * bits // 8)
            assert np.array_equal(O.unpack_codes(p, bits, d), c)


# --------------------------------------------------------------------------
# Per-channel key quantization over token blocks (section 2: KIVI-style
# per-channel keys; Eq. (1) per group)
# --------------------------------------------------------------------------


def check_key_channel_hand_fixture():
    for line in _rows("key_channel.txt"):
        parts = [p.strip() for p in line.split("|")]
        bits = int(parts[0])
        y = np.array([[float(v) for v in t.split()] for t in parts[1].split(";")], dtype=np.float32)
        d_want = np.array([float(v) for v in parts[2].split()])
        z_want = np.array([float(v) for v in parts[3].split()])
        c_want = np.array([[int(v) for v in t.split()] for t in parts[4].split(";")])
        codes, delta, zero = O.quantize_key_channels(y, bits)
        assert np.array_equal(delta[0], d_want.astype(np.float32)), (line, delta)
        assert np.array_equal(zero[0], z_want.astype(np.float32)), (line, zero)
        assert np.array_equal(codes, c_want), (line, codes)
        xh = O.dequantize_key_channels(codes, delta, zero)
        assert np.array_equal(xh, (c_want - z_want[None]) * d_want[None])


def check_key_channel_blocks():
    """Blocks of 128 tokens from each chunk's first token (the last one
    shorter); a block's steps, zero points and codes depend on its own
    tokens only; every unclamped element within half a step, every code the
    nearest grid point of its channel (brute force over all codes)."""
    assert O.chunk_blocks(300) == [(0, 128), (128, 256), (256, 300)]
    assert O.chunk_blocks(128) == [(0, 128)]
    assert O.chunk_blocks(1) == [(0, 1)]
    rng = np.random.default_rng(21)
    for bits in (2, 4):
        y = (rng.standard_normal((300, 64)) * rng.uniform(0.2, 4, (1, 64))
             + rng.standard_normal((1, 64))).astype(np.float32)
        codes, delta, zero = O.quantize_key_channels(y, bits)
        assert delta.shape == (3, 64) and codes.shape == (300, 64)
        y2 = y.copy()
        y2[5] *= 7.0                                 # a token of block 0 only
        c2, d2, z2 = O.quantize_key_channels(y2, bits)
        assert np.array_equal(c2[128:], codes[128:]) and np.array_equal(d2[1:], delta[1:])
        assert not np.array_equal(d2[0], delta[0])
        qmax = 2 ** bits - 1
        dl = O.key_channel_token_steps(delta.astype(np.float64), 300)
        zz = O.key_channel_token_steps(zero.astype(np.float64), 300)
        xh = O.dequantize_key_channels(codes, delta, zero)
        err = np.abs(xh - y)
        unclamped = (codes > 0) & (codes < qmax)
        assert np.all(err[unclamped] <= dl[unclamped] / 2 * (1 + 1e-6))
        cands = (np.arange(qmax + 1)[None, None, :] - zz[..., None]) * dl[..., None]
        best = np.abs(cands - y[..., None].astype(np.float64)).min(axis=-1)
        assert np.all(err <= best + 1e-6 * dl)
        # per channel, the step covers the block's range (BF16 rounding aside)
        for i, (a, b) in enumerate(O.chunk_blocks(300)):
            rng_c = y[a:b].max(0).astype(np.float64) - y[a:b].min(0)
            assert np.all(np.abs(delta[i] - rng_c / qmax) <= delta[i] * 2 ** -8 + 1e-30)


def check_key_channel_bias_brute_force():
    """With per-channel key steps the correction keeps its form with one
    channel per group: b_Taylor = scale^2 / 24 * sum_c q'_c^2 D_c^2 and
    b_exact = sum_c log(sinh a_c / a_c), a_c = scale |q'_c| D_c / 2, D_c the
    step of the key's block in channel c (loops, fp64)."""
    rng = np.random.default_rng(22)
    d, scale = 8, 0.35
    q = rng.standard_normal((3, d))
    dl = rng.uniform(0.05, 1.5, (4, d))
    bt = O.jensen_bias_taylor(q, dl, scale, 1)
    be = O.jensen_bias_exact(q, dl, scale, 1)
    for j in range(3):
        for i in range(4):
            t = sum(scale * scale / 24 * q[j, c] ** 2 * dl[i, c] ** 2 for c in range(d))
            e = 0.0
            for c in range(d):
                a = 0.5 * scale * abs(q[j, c]) * dl[i, c]
                e += math.log(math.sinh(a) / a)
            assert abs(bt[j, i] - t) <= 1e-14 * abs(t)
            assert abs(be[j, i] - e) <= 1e-12 * abs(e)


def check_key_channel_mass_shift():
    """The per-channel key scheme shows the same Jensen effect (Figure 2 /
    section 1: quantized keys take mass from the current chunk) and the same
    correction, with per-channel steps, undoes most of it (section 2: the
    correction is orthogonal to the quantization scheme)."""
    rng = np.random.default_rng(23)
    d, n_q, n_r, chunk, n_chunks, scale = 64, 256, 256, 256, 4, 1 / 8
    s = np.where(rng.integers(0, 2, d) == 1, -1.0, 1.0).astype(np.float32)
    q = O.bf16_round(rng.standard_normal((n_q, d)).astype(np.float32))
    kc = O.bf16_round(rng.standard_normal((n_r, d)).astype(np.float32))
    vc = O.bf16_round(rng.standard_normal((n_r, d)).astype(np.float32))
    k = rng.standard_normal((chunk * n_chunks, d)).astype(np.float32)
    k[:, :4] *= 8
    k = O.bf16_round(k)
    v = O.bf16_round(rng.standard_normal((chunk * n_chunks, d)).astype(np.float32))
    kh, steps = [], []
    for c0 in range(0, k.shape[0], chunk):
        _, kd, kz, _, codes = O.quantize_key_chunk(k[c0:c0 + chunk], s, 2)
        kh.append(O.dequantize_key_channels(codes, kd, kz))
        steps.append(O.key_channel_token_steps(kd, chunk))
    kh = np.concatenate(kh)
    steps = np.concatenate(steps)
    vr = O.rotate(v, s)
    _, ps_ref, _ = O.chunk_attention(q, O.rotate(k, s), vr, np.zeros((k.shape[0], 1)), kc, vc, s,
                                     scale, 1, O.CORR_NONE)
    ps = {c: O.chunk_attention(q, kh, vr, steps, kc, vc, s, scale, 1, c)[1]
          for c in (O.CORR_NONE, O.CORR_TAYLOR, O.CORR_EXACT)}
    shift = ps[O.CORR_NONE].mean() - ps_ref.mean()
    assert shift > 1e-2
    assert abs(ps[O.CORR_TAYLOR].mean() - ps_ref.mean()) < 0.25 * shift
    assert abs(ps[O.CORR_EXACT].mean() - ps_ref.mean()) < 0.25 * shift


# --------------------------------------------------------------------------
# Jensen bias (Figure 3 caption; abstract; section 1)
# --------------------------------------------------------------------------


def check_log_sinhc_closed_form():
    import mpmath as mp
    mp.mp.dps = 40
    a = np.array([1e-6, 1e-4, 5e-4, 1e-3, 2e-3, 0.01, 0.1, 0.5, 0.999, 1.0, 2.0, 7.0, 30.0])
    want = np.array([float(mp.log(mp.sinh(mp.mpf(v)) / mp.mpf(v))) for v in a])
    got = O.log_sinhc(a)
    assert np.all(np.abs(got - want) <= 1e-14 * np.abs(want)), (got, want)
    assert abs(O.log_sinhc(np.array([1.0]))[0] - 0.161439362) < 1e-9
    assert abs(O.log_sinhc(np.array([0.5]))[0] - 0.041324855) < 1e-9


def check_bias_forms():
    """b_Taylor = sum_c a_c^2 / 6 (a_c = scale |q'_c| D_g(c) / 2), the
    second-order term of b_exact = sum_c log(sinh a_c / a_c); the gap is
    -sum a^4 / 180 to leading order; D -> 0 gives b = 0."""
    rng = np.random.default_rng(7)
    d, group, scale = 64, 16, 1 / 8
    q = rng.standard_normal((6, d))
    dl = rng.uniform(0.01, 0.05, (9, d // group))
    bt = O.jensen_bias_taylor(q, dl, scale, group)
    a = 0.5 * scale * np.abs(q)[:, None, :] * np.repeat(dl, group, axis=1)[None, :, :]
    assert np.allclose(bt, (a ** 2).sum(-1) / 6, rtol=1e-12, atol=0)
    be = O.jensen_bias_exact(q, dl, scale, group)
    assert np.allclose(be - bt, -(a ** 4).sum(-1) / 180, rtol=2e-3, atol=1e-18)
    assert np.all(be < bt)   # the Taylor term over-corrects slightly
    z = np.zeros_like(dl)
    assert np.all(O.jensen_bias_taylor(q, z, scale, group) == 0)
    assert np.all(O.jensen_bias_exact(q, z, scale, group) == 0)


def check_monte_carlo_jensen():
    """Figure 3: uniform zero-mean noise leaves s_hat unbiased, inflates
    E[exp(s_hat)] above exp(s); subtracting b_exact removes that in
    expectation, and b_Taylor nearly so (O(a^4))."""
    rng = np.random.default_rng(8)
    d, group, scale = 32, 32, 1 / math.sqrt(32)
    q = rng.standard_normal((1, d)) * 1.5
    delta = np.array([[1.2]])
    n = 400_000
    eps = (rng.random((n, d)) - 0.5) * delta[0, 0]
    noise = scale * (eps @ q[0])                      # s_hat - s per draw
    se = noise.std() / math.sqrt(n)
    assert abs(noise.mean()) < 5 * se                 # unbiased score
    var_pred = scale ** 2 * (q[0] ** 2).sum() * delta[0, 0] ** 2 / 12
    assert abs(noise.var() / var_pred - 1) < 0.02
    e = np.exp(noise)
    se_e = e.std() / math.sqrt(n)
    jensen = e.mean() - 1.0
    assert jensen > 20 * se_e                         # E[e^s_hat] > e^s
    b_ex = O.jensen_bias_exact(q, delta, scale, group)[0, 0]
    b_ty = O.jensen_bias_taylor(q, delta, scale, group)[0, 0]
    assert abs(b_ty - var_pred / 2) < 1e-12
    r_ex = np.exp(noise - b_ex).mean() - 1.0
    r_ty = np.exp(noise - b_ty).mean() - 1.0
    assert abs(r_ex) < 5 * se_e
    assert abs(r_ty) < abs(jensen) / 5
    a4 = ((0.5 * scale * np.abs(q[0]) * delta[0, 0]) ** 4).sum() / 180
    assert abs(r_ty) < 2 * a4 + 5 * se_e


# --------------------------------------------------------------------------
# Attention and masses
# --------------------------------------------------------------------------


def _brute_attention(q, ks_rot, vs_rot, dl, kc, vc, signs, scale, group, corr):
    """Pure-Python loops, fp64, tiny sizes only."""
    d = len(signs)
    r = O.rotation_matrix(signs)
    out, ps, pr = [], [], []
    for qj in q:
        qr = [sum(r[a][c] * qj[c] for c in range(d)) for a in range(d)]
        scores = []
        for i, ki in enumerate(ks_rot):
            s = scale * sum(qr[c] * ki[c] for c in range(d))
            if corr == O.CORR_TAYLOR:
                b = 0.0
                for c in range(d):
                    b += (scale * qr[c] * dl[i][c // group]) ** 2 / 24
                s -= b
            elif corr == O.CORR_EXACT:
                b = 0.0
                for c in range(d):
                    a = 0.5 * scale * abs(qr[c]) * dl[i][c // group]
                    b += math.log(math.sinh(a) / a) if a > 0 else 0.0
                s -= b
            scores.append(s)
        for ki in kc:
            scores.append(scale * sum(qj[c] * ki[c] for c in range(d)))
        m = max(scores)
        e = [math.exp(s - m) for s in scores]
        tot = sum(e)
        p = [x / tot for x in e]
        ns = len(ks_rot)
        ps.append(sum(p[:ns]))
        pr.append(sum(p[ns:]))
        vals = [[sum(r[a][c] * vi[a] for a in range(d)) for c in range(d)] for vi in vs_rot]
        vals += [list(v) for v in vc]
        out.append([sum(p[i] * vals[i][c] for i in range(len(p))) for c in range(d)])
    return np.array(out), np.array(ps), np.array(pr)


def check_attention_brute_force():
    rng = np.random.default_rng(9)
    d, group, scale = 4, 2, 0.5
    s = np.array([1.0, -1.0, -1.0, 1.0])
    q = rng.standard_normal((3, d))
    ks = rng.standard_normal((5, d))
    vs = rng.standard_normal((5, d))
    dl = rng.uniform(0.2, 0.9, (5, d // group))
    kc = rng.standard_normal((2, d))
    vc = rng.standard_normal((2, d))
    for corr in (O.CORR_NONE, O.CORR_TAYLOR, O.CORR_EXACT):
        o, ps, pr = O.chunk_attention(q, ks, vs, dl, kc, vc, s, scale, group, corr)
        ob, psb, prb = _brute_attention(q, ks, vs, dl, kc, vc, s, scale, group, corr)
        assert np.allclose(o, ob, rtol=0, atol=1e-12)
        assert np.allclose(ps, psb, rtol=0, atol=1e-13)
        assert np.allclose(pr, prb, rtol=0, atol=1e-13)
        assert np.allclose(ps + pr, 1.0, atol=1e-14)


def _sdpa(q, k, v, scale):
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))[None, None]
    return torch.nn.functional.scaled_dot_product_attention(
        t(q), t(k), t(v), scale=scale)[0, 0].numpy()


def check_attention_special_cases():
    """Empty cache = textbook softmax attention over the current chunk; a
    rotated cache with zero step sizes (b = 0) = textbook attention over the
    union of cached and current tokens, in the original basis."""
    rng = np.random.default_rng(10)
    d, group, scale = 64, 32, 1 / 8
    s = np.where(rng.integers(0, 2, d) == 1, -1.0, 1.0)
    q = rng.standard_normal((17, d))
    kc = rng.standard_normal((11, d))
    vc = rng.standard_normal((11, d))
    e = np.zeros((0, d))
    o, ps, pr = O.chunk_attention(q, e, e, np.zeros((0, 2)), kc, vc, s, scale, group)
    assert np.allclose(o, _sdpa(q, kc, vc, scale), atol=1e-12)
    assert np.all(ps == 0) and np.allclose(pr, 1.0, atol=1e-14)
    k = rng.standard_normal((13, d))
    v = rng.standard_normal((13, d))
    for corr in (O.CORR_NONE, O.CORR_TAYLOR, O.CORR_EXACT):
        o, ps, pr = O.chunk_attention(q, O.rotate(k, s), O.rotate(v, s), np.zeros((13, 2)),
                                      kc, vc, s, scale, group, corr)
        want = _sdpa(q, np.concatenate([k, kc]), np.concatenate([v, vc]), scale)
        assert np.allclose(o, want, atol=1e-12)
    o, ps, pr = O.chunk_attention(q, O.rotate(k, s), O.rotate(v, s), np.zeros((13, 2)),
                                  e, e, s, scale, group)
    assert np.allclose(ps, 1.0, atol=1e-14) and np.all(pr == 0)
    assert np.allclose(o, _sdpa(q, k, v, scale), atol=1e-12)


def _quantized_head(bits, group, seed=11, n_q=256, n_s=1024, n_r=256, d=64):
    rng = np.random.default_rng(seed)
    s = np.where(rng.integers(0, 2, d) == 1, -1.0, 1.0).astype(np.float32)
    q = O.bf16_round(rng.standard_normal((n_q, d)).astype(np.float32))
    kc = O.bf16_round(rng.standard_normal((n_r, d)).astype(np.float32))
    vc = O.bf16_round(rng.standard_normal((n_r, d)).astype(np.float32))
    k = rng.standard_normal((n_s, d)).astype(np.float32)
    k[:, :4] *= 8
    k = O.bf16_round(k)
    v = O.bf16_round(rng.standard_normal((n_s, d)).astype(np.float32))
    _, kd, kz, _, kcodes = O.quantize_rows(k, s, bits, group)
    _, vd, vz, _, vcodes = O.quantize_rows(v, s, bits, group)
    qd = dict(kh=O.dequantize(kcodes, kd, kz, group), vh=O.dequantize(vcodes, vd, vz, group),
              kd=kd)
    return q, k, v, kc, vc, s, qd


def check_mass_shift_and_correction():
    """Figure 2 / Figure 4 / section 1: with an INT2 cache, attention mass
    moves to the cached block (P_S grows) relative to unquantized keys, and
    the correction brings P_S back toward the unquantized value.  Direction
    only: the paper prints no magnitudes."""
    q, k, v, kc, vc, s, qd = _quantized_head(2, 32)
    scale = 1 / 8
    _, ps_ref, _ = O.chunk_attention(q, O.rotate(k, s), O.rotate(v, s), np.zeros((k.shape[0], 2)),
                                     kc, vc, s, scale, 32, O.CORR_NONE)
    _, ps_q, _ = O.chunk_attention(q, qd["kh"], qd["vh"], qd["kd"], kc, vc, s, scale, 32, O.CORR_NONE)
    _, ps_c, _ = O.chunk_attention(q, qd["kh"], qd["vh"], qd["kd"], kc, vc, s, scale, 32, O.CORR_TAYLOR)
    _, ps_e, _ = O.chunk_attention(q, qd["kh"], qd["vh"], qd["kd"], kc, vc, s, scale, 32, O.CORR_EXACT)
    shift = ps_q.mean() - ps_ref.mean()
    assert shift > 1e-3
    assert abs(ps_c.mean() - ps_ref.mean()) < 0.5 * shift
    assert abs(ps_e.mean() - ps_ref.mean()) < 0.5 * shift
    assert np.mean(ps_q > ps_ref) > 0.8


def check_int4_beats_int2_uncorrected():
    """Section 1: INT4 keeps reasonable quality, INT2 distorts far more --
    here, the attention output error against unquantized keys/values."""
    errs = {}
    for bits, group in ((2, 32), (4, 64)):
        q, k, v, kc, vc, s, qd = _quantized_head(bits, group)
        o_ref, _, _ = O.chunk_attention(q, O.rotate(k, s), O.rotate(v, s),
                                        np.zeros((k.shape[0], 2)), kc, vc, s, 1 / 8, 32)
        o, _, _ = O.chunk_attention(q, qd["kh"], qd["vh"], qd["kd"], kc, vc, s, 1 / 8, group,
                                    O.CORR_NONE)
        errs[bits] = np.abs(o - o_ref).mean()
    assert errs[4] < errs[2] / 2, errs


def check_ring_rules():
    C, n = 10, 3
    assert O.ring_append(0, 0, 10, C, n) == (0, 10, 1)
    assert O.ring_append(10, 1, 10, C, n) == (10, 20, 2)
    assert O.ring_append(20, 2, 4, C, n) == (20, 24, 0)        # partial newest chunk
    assert O.ring_append(24, 0, 10, C, n) is None               # nothing after a partial one
    assert O.ring_append(20, 2, 10, C, n) == (20, 30, 0)
    assert O.ring_append(30, 0, 10, C, n) == (0, 30, 1)         # wrap: overwrite oldest
    assert O.ring_append(30, 1, 9, C, n) is None                # full: whole chunks only
    assert O.ring_append(30, 1, 0, C, n) == (10, 30, 1)
    assert O.ring_append(0, 0, 11, C, n) is None


ALL_CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]
