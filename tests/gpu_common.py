"""Shared helpers of the GPU parity tests: build a cache through the C-ABI,
and compute the oracle's answer from the same seeded BF16 inputs (never from
anything the CUDA path produced)."""
from __future__ import annotations

import numpy as np

from oracle import kvq_oracle as O
from quantized_kv_cache_quantize_gb300 import kvq, synth

O_TOL = 2e-2      # max-abs error of O, relative to max |O_ref| over compared rows
MASS_TOL = 1e-3   # absolute error of P_S, P_R per row


def build_cache(w: synth.Workload, x: dict, signs, n_s: int | None = None) -> kvq.KVCache:
    """Quantize-append the window k_win/v_win chunk by chunk (the last chunk
    may be partial)."""
    n_s = x["k_win"].shape[-2] if n_s is None else n_s
    cache = kvq.KVCache(x["k_win"].shape[0], x["k_win"].shape[1], w.head_dim, w.bits, w.group,
                        w.chunk_tokens, w.n_chunks, signs)
    kw = x["k_win"].cuda()
    vw = x["v_win"].cuda()
    for c0 in range(0, n_s, w.chunk_tokens):
        c1 = min(n_s, c0 + w.chunk_tokens)
        kvq.quantize_append(cache, kw[:, :, c0:c1].contiguous(), vw[:, :, c0:c1].contiguous())
    return cache


def oracle_head(w: synth.Workload, x: dict, signs, b: int, h: int, rows, corr: int,
                n_s: int | None = None):
    """Oracle O, P_S, P_R of query rows ``rows`` of head (b, h)."""
    n_s = x["k_win"].shape[-2] if n_s is None else n_s
    kf = x["k_win"][b, h, :n_s].float().numpy()
    vf = x["v_win"][b, h, :n_s].float().numpy()
    _, kd, kz, _, kc = O.quantize_rows(kf, signs, w.bits, w.group)
    _, vd, vz, _, vc = O.quantize_rows(vf, signs, w.bits, w.group)
    q = x["q"][b, h].float().numpy()[rows]
    return O.chunk_attention(q, O.dequantize(kc, kd, kz, w.group), O.dequantize(vc, vd, vz, w.group),
                             kd, x["k_cur"][b, h].float().numpy(), x["v_cur"][b, h].float().numpy(),
                             signs, w.scale, w.group, corr)


def admissible(x, signs, bits: int, group: int, packed, sz_bits):
    """Check packed codes and (step, zero) BF16 bits [..., G, 2] that the
    GPU wrote for BF16 rows x [..., d] against every answer the oracle
    allows: the rotation known to within its fp32 summation bound
    (O.rotation_bounds; exact for rows whose partial sums are all fp32
    numbers) and Eq. (1) over that interval (O.quantize_groups_admissible).
    Returns (per-group bool: the GPU's step, zero point and codes form one
    admissible answer; the fraction of codes the bounds determine)."""
    xf = x.float().numpy() if hasattr(x, "float") else np.asarray(x, np.float32)
    lo, hi = O.rotation_bounds(xf, signs)
    cd, cz, clo, chi = O.quantize_groups_admissible(lo, hi, bits, group)
    d = xf.shape[-1]
    lead = xf.shape[:-1]
    codes = O.unpack_codes(packed, bits, d).reshape(*lead, d // group, group)
    sz = np.asarray(sz_bits).view(np.uint16)
    ok = ((O.bf16_bits(cd) == sz[..., 0][..., None]) & (O.bf16_bits(cz) == sz[..., 1][..., None]) &
          np.all((clo <= codes[..., None, :]) & (codes[..., None, :] <= chi), axis=-1))
    return ok.any(axis=-1), float(np.mean(clo == chi))


def assert_close(o_gpu, o_ref, ps_gpu=None, ps_ref=None, pr_gpu=None, pr_ref=None, what=""):
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    err = np.abs(o_gpu - o_ref).max()
    ref = np.abs(o_ref).max()
    assert np.all(np.isfinite(o_gpu)), what
    assert err <= O_TOL * ref, f"{what}: max|dO| {err:.4g} > {O_TOL} * {ref:.4g}"
    if ps_gpu is not None:
        e_s = np.abs(np.asarray(ps_gpu, np.float64) - ps_ref).max()
        e_r = np.abs(np.asarray(pr_gpu, np.float64) - pr_ref).max()
        assert e_s <= MASS_TOL and e_r <= MASS_TOL, f"{what}: mass err {e_s:.3g} {e_r:.3g}"
    return err / ref


def build_cache_kch(w: synth.Workload, x: dict, signs, n_s: int | None = None) -> kvq.KVCache:
    """As build_cache, with per-channel key quantization."""
    n_s = x["k_win"].shape[-2] if n_s is None else n_s
    cache = kvq.KVCache(x["k_win"].shape[0], x["k_win"].shape[1], w.head_dim, w.bits, w.group,
                        w.chunk_tokens, w.n_chunks, signs, key_mode=kvq.KEYS_PER_CHANNEL)
    kw = x["k_win"].cuda()
    vw = x["v_win"].cuda()
    for c0 in range(0, n_s, w.chunk_tokens):
        c1 = min(n_s, c0 + w.chunk_tokens)
        kvq.quantize_append(cache, kw[:, :, c0:c1].contiguous(), vw[:, :, c0:c1].contiguous())
    return cache


def oracle_head_kch(w: synth.Workload, x: dict, signs, b: int, h: int, rows, corr: int,
                    n_s: int | None = None):
    """Oracle O, P_S, P_R with per-channel keys: each appended chunk's keys
    quantized per channel over 128-token blocks, the correction with one
    channel per group (the key's block steps)."""
    n_s = x["k_win"].shape[-2] if n_s is None else n_s
    kf = x["k_win"][b, h, :n_s].float().numpy()
    vf = x["v_win"][b, h, :n_s].float().numpy()
    kh, steps = [], []
    for c0 in range(0, n_s, w.chunk_tokens):
        part = kf[c0:c0 + w.chunk_tokens]
        _, kd, kz, _, kc = O.quantize_key_chunk(part, signs, w.bits)
        kh.append(O.dequantize_key_channels(kc, kd, kz))
        steps.append(O.key_channel_token_steps(kd, part.shape[0]))
    d = kf.shape[1]
    kh = np.concatenate(kh) if kh else np.zeros((0, d))
    steps = np.concatenate(steps) if steps else np.zeros((0, d))
    _, vd, vz, _, vc = O.quantize_rows(vf, signs, w.bits, w.group)
    q = x["q"][b, h].float().numpy()[rows]
    return O.chunk_attention(q, kh, O.dequantize(vc, vd, vz, w.group), steps,
                             x["k_cur"][b, h].float().numpy(), x["v_cur"][b, h].float().numpy(),
                             signs, w.scale, 1, corr)
