"""GPU parity of the per-channel key mode (KIVI-style keys: per channel over
128-token blocks of each chunk, values per token and group) against the
oracle, through the C-ABI: O within 2e-2 x max|O_ref|, P_S and P_R within
1e-3 per row, for every correction mode."""
import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O
from quantized_kv_cache_quantize_gb300 import kvq, synth
from tests.gpu_common import assert_close, build_cache_kch, oracle_head_kch

pytestmark = pytest.mark.gpu

CORRS = [kvq.CORR_TAYLOR, kvq.CORR_NONE, kvq.CORR_EXACT]


@pytest.mark.parametrize("corr", CORRS)
def test_tiny_all_rows(corr):
    w = synth.WORKLOADS["tiny"]
    x = synth.inputs(w)
    s = synth.hadamard_signs(w.head_dim)
    cache = build_cache_kch(w, x, s)
    out, ps, pr = kvq.attention_corrected(cache, x["q"].cuda(), x["k_cur"].cuda(),
                                          x["v_cur"].cuda(), corr=corr, with_mass=True)
    torch.cuda.synchronize()
    assert kvq.last_device_status() == 0
    o_ref, ps_ref, pr_ref = oracle_head_kch(w, x, s, 0, 0, np.arange(w.n_q), corr)
    assert_close(out[0, 0].float().cpu().numpy(), o_ref, ps[0, 0].cpu().numpy(), ps_ref,
                 pr[0, 0].cpu().numpy(), pr_ref, what=f"tiny per-channel corr={corr}")
    ps2, pr2 = kvq.attention_mass(cache, x["q"].cuda(), x["k_cur"].cuda(), corr=corr)
    assert torch.allclose(ps2, ps, atol=1e-6) and torch.allclose(pr2, pr, atol=1e-6)


RAGGED = [
    # (d, bits, group, n_q, n_s, n_r, chunk, n_chunks, heads)
    (128, 2, 32, 300, 900, 300, 300, 3, 2),     # blocks 128, 128, 44 per chunk
    (128, 2, 32, 129, 650, 77, 300, 3, 1),      # a partial last chunk (50 tokens)
    (64, 2, 32, 1, 1, 1, 1, 1, 1),
    (64, 4, 64, 200, 256, 0, 128, 2, 2),        # chunks of exactly one block
    (128, 4, 64, 257, 130, 257, 65, 2, 1),      # chunks shorter than a block
    (128, 2, 64, 100, 0, 90, 50, 2, 1),         # empty cache
]


@pytest.mark.parametrize("case", RAGGED, ids=lambda c: "d{}b{}g{}_q{}_s{}_r{}_c{}".format(*c[:7]))
@pytest.mark.parametrize("corr,flags", [
    (kvq.CORR_TAYLOR, 0), (kvq.CORR_NONE, kvq.FLAG_NO_KV_SPLIT),
    (kvq.CORR_EXACT, 0), (kvq.CORR_TAYLOR, kvq.FLAG_PRECISE_QUERY | kvq.FLAG_NO_KV_SPLIT)])
def test_ragged_all_rows(case, corr, flags):
    """Chunks that are not multiples of the 128-token block, partial chunks,
    single tokens, an empty cache; with and without the key-range split."""
    d, bits, group, n_q, n_s, n_r, chunk, n_chunks, heads = case
    w = synth.Workload("kch", heads=heads, head_dim=d, chunk_tokens=chunk, n_chunks=n_chunks,
                       bits=bits, group=group, n_outliers_fixed=2, outlier_scale=6.0,
                       offset_std=0.3)
    x = synth.inputs(w, n_q=n_q, n_s=n_s, n_r=n_r)
    s = synth.hadamard_signs(d, seed=3)
    cache = build_cache_kch(w, x, s, n_s=n_s)
    assert cache.len == n_s
    out, ps, pr = kvq.attention_corrected(cache, x["q"].cuda(), x["k_cur"].cuda(),
                                          x["v_cur"].cuda(), corr=corr, with_mass=True,
                                          flags=flags)
    torch.cuda.synchronize()
    assert kvq.last_device_status() == 0
    for h in range(heads):
        o_ref, ps_ref, pr_ref = oracle_head_kch(w, x, s, 0, h, np.arange(n_q), corr, n_s=n_s)
        assert_close(out[0, h].float().cpu().numpy(), o_ref, ps[0, h].cpu().numpy(), ps_ref,
                     pr[0, h].cpu().numpy(), pr_ref, what=f"{case} h{h}")


def test_correction_restores_mass():
    """Figure 2 / section 1 with per-channel keys (section 2: the correction
    is orthogonal to the quantization scheme): quantized keys raise P_S over
    unquantized keys and both corrections bring it back."""
    w = synth.WORKLOADS["tiny"]
    x = synth.inputs(w)
    s = synth.hadamard_signs(w.head_dim)
    cache = build_cache_kch(w, x, s)
    q, kc = x["q"].cuda(), x["k_cur"].cuda()
    ps = {c: kvq.attention_mass(cache, q, kc, corr=c)[0].mean().item() for c in CORRS}
    kf = x["k_win"][0, 0].float().numpy()
    _, ps_ref, _ = O.chunk_attention(x["q"][0, 0].float().numpy(), O.rotate(kf, s),
                                     O.rotate(x["v_win"][0, 0].float().numpy(), s),
                                     np.zeros((kf.shape[0], 1)), x["k_cur"][0, 0].float().numpy(),
                                     x["v_cur"][0, 0].float().numpy(), s, w.scale, 1, O.CORR_NONE)
    shift = ps[kvq.CORR_NONE] - ps_ref.mean()
    assert shift > 0.01
    assert abs(ps[kvq.CORR_TAYLOR] - ps_ref.mean()) < 0.25 * shift
    assert abs(ps[kvq.CORR_EXACT] - ps_ref.mean()) < 0.25 * shift


@pytest.mark.parametrize("name,corr,flags,heads,rows", [
    ("w4_int2", kvq.CORR_TAYLOR, 0, 24, 48),
    ("w4_int2", kvq.CORR_EXACT, 0, 4, 32),
    ("hires_t3", kvq.CORR_TAYLOR, kvq.FLAG_PRECISE_QUERY, 6, 32)])
def test_full_workload_sampled_rows(name, corr, flags, heads, rows):
    """Full-size workloads in the per-channel key mode (the launch
    configuration of ``bench.py --keys channel``): sampled heads and rows."""
    w = synth.WORKLOADS[name]
    x = synth.inputs(w)
    s = synth.hadamard_signs(w.head_dim)
    cache = build_cache_kch(w, x, s)
    out, ps, pr = kvq.attention_corrected(cache, x["q"].cuda(), x["k_cur"].cuda(),
                                          x["v_cur"].cuda(), corr=corr, with_mass=True, flags=flags)
    torch.cuda.synchronize()
    assert kvq.last_device_status() == 0
    rng = np.random.default_rng(13)
    hs = range(w.heads) if heads >= w.heads else rng.choice(w.heads, heads, replace=False)
    for h in hs:
        sel = np.unique(np.concatenate([[0, w.n_q - 1], rng.choice(w.n_q, rows - 2, replace=False)]))
        o_ref, ps_ref, pr_ref = oracle_head_kch(w, x, s, 0, int(h), sel, corr)
        assert_close(out[0, h, sel].float().cpu().numpy(), o_ref, ps[0, h, sel].cpu().numpy(),
                     ps_ref, pr[0, h, sel].cpu().numpy(), pr_ref, what=f"{name} kch h{h}")


def test_batch_and_heads_layout():
    """batch 2 x heads 3 with per-channel keys: each (b, h) attends to its own
    cache (its own per-block steps) and chunk."""
    w = synth.Workload("kch_bh", heads=3, head_dim=128, chunk_tokens=200, n_chunks=2, bits=2,
                       group=32, n_outliers_fixed=3, outlier_scale=10.0, offset_std=0.5)
    xs = [synth.inputs(w, seed=sd, n_q=150, n_s=400, n_r=90) for sd in (1, 2)]
    x = {k: torch.cat([xs[0][k], xs[1][k]], dim=0).contiguous() for k in xs[0]}
    s = synth.hadamard_signs(128, seed=5)
    cache = build_cache_kch(w, x, s)
    out, ps, pr = kvq.attention_corrected(cache, x["q"].cuda(), x["k_cur"].cuda(),
                                          x["v_cur"].cuda(), with_mass=True)
    torch.cuda.synchronize()
    for b in range(2):
        for h in range(3):
            o_ref, ps_ref, pr_ref = oracle_head_kch(w, x, s, b, h, np.arange(150), O.CORR_TAYLOR)
            assert_close(out[b, h].float().cpu().numpy(), o_ref, ps[b, h].cpu().numpy(), ps_ref,
                         pr[b, h].cpu().numpy(), pr_ref, what=f"kch b{b} h{h}")


@pytest.mark.parametrize("corr", CORRS)
def test_noalloc_matches_workspace(corr):
    """The allocation-free entry point with per-channel keys (its built-in
    scratch also holds the per-(row, tile) table) gives what the workspace
    entry point gives."""
    w = synth.Workload("kch_na", heads=2, head_dim=128, chunk_tokens=300, n_chunks=3, bits=2,
                       group=32, n_outliers_fixed=3, outlier_scale=8.0, offset_std=0.4)
    x = synth.inputs(w, seed=31, n_q=400, n_s=900, n_r=300)
    s = synth.hadamard_signs(128, seed=31)
    cache = build_cache_kch(w, x, s)
    q, kc, vc = x["q"].cuda(), x["k_cur"].cuda(), x["v_cur"].cuda()
    ref_o, ref_ps, _ = kvq.attention_corrected(cache, q, kc, vc, corr=corr, with_mass=True)
    o, ps, _ = kvq.attention_corrected_noalloc(cache, q, kc, vc, corr=corr, with_mass=True)
    torch.cuda.synchronize()
    assert kvq.last_device_status() == kvq.KVQ_OK
    ref = ref_o.float()
    assert (o.float() - ref).abs().max().item() <= 2e-2 * ref.abs().max().item()
    assert (ps - ref_ps).abs().max().item() <= 1e-3
