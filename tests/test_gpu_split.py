"""GPU parity of the key-range split: when the (head, query block) grid would
leave most SMs idle, each CTA takes one contiguous range of key tiles, leaves
its unnormalized O', base and partial sums, and a merge kernel combines the
ranges (the online-softmax combination of disjoint key sets, then the inverse
rotation).  Few queries over long windows, every row against the oracle and
against the unsplit kernel (FLAG_NO_KV_SPLIT)."""
import numpy as np
import pytest
import torch

from quantized_kv_cache_quantize_gb300 import kvq, synth
from tests.gpu_common import assert_close, build_cache, oracle_head

pytestmark = pytest.mark.gpu

SPLIT = [
    # (d, bits, group, n_q, n_s, n_r, chunk, n_chunks, heads)
    (128, 2, 32, 1, 3000, 100, 1000, 3, 2),      # one query row per head
    (128, 4, 64, 60, 4096, 128, 1024, 4, 1),     # 33 tiles, 16-way bound
    (64, 2, 32, 130, 2500, 300, 500, 5, 3),      # ragged ranges, d = 64
    (128, 2, 64, 256, 5000, 256, 1000, 5, 1),    # range boundary inside the current chunk
    (128, 2, 32, 77, 0, 1500, 500, 2, 2),        # current chunk only
]


def _setup(case, seed=5):
    d, bits, group, n_q, n_s, n_r, chunk, n_chunks, heads = case
    w = synth.Workload("split", heads=heads, head_dim=d, chunk_tokens=chunk, n_chunks=n_chunks,
                       bits=bits, group=group, n_outliers_fixed=2, outlier_scale=6.0,
                       offset_std=0.3)
    x = synth.inputs(w, seed=seed, n_q=n_q, n_s=n_s, n_r=n_r)
    s = synth.hadamard_signs(d, seed=11)
    cache = build_cache(w, x, s, n_s=n_s)
    assert cache.len == n_s
    return w, x, s, cache


@pytest.mark.parametrize("case", SPLIT, ids=lambda c: "d{}b{}g{}_q{}_s{}_r{}".format(*c[:6]))
@pytest.mark.parametrize("corr,flags", [(kvq.CORR_TAYLOR, 0), (kvq.CORR_NONE, 0),
                                        (kvq.CORR_TAYLOR, kvq.FLAG_PRECISE_QUERY)])
def test_split_all_rows(case, corr, flags):
    w, x, s, cache = _setup(case)
    n_q, n_s, heads = case[3], case[4], case[8]
    q, kc, vc = x["q"].cuda(), x["k_cur"].cuda(), x["v_cur"].cuda()
    out, ps, pr = kvq.attention_corrected(cache, q, kc, vc, corr=corr, with_mass=True, flags=flags)
    torch.cuda.synchronize()
    assert kvq.last_device_status() == 0
    for h in range(heads):
        o_ref, ps_ref, pr_ref = oracle_head(w, x, s, 0, h, np.arange(n_q), corr, n_s=n_s)
        assert_close(out[0, h].float().cpu().numpy(), o_ref, ps[0, h].cpu().numpy(), ps_ref,
                     pr[0, h].cpu().numpy(), pr_ref, what=f"{case} h{h}")
    # the unsplit kernel on the same inputs: the two differ only by the FP16
    # rounding of P against different bases
    out1, ps1, pr1 = kvq.attention_corrected(cache, q, kc, vc, corr=corr, with_mass=True,
                                             flags=flags | kvq.FLAG_NO_KV_SPLIT)
    torch.cuda.synchronize()
    assert kvq.last_device_status() == 0
    ref = out1.float().abs().max().item()
    assert (out.float() - out1.float()).abs().max().item() <= 1e-2 * ref
    assert (ps - ps1).abs().max().item() <= 5e-4 and (pr - pr1).abs().max().item() <= 5e-4
    # the mass-only entry point takes the same split
    ps2, pr2 = kvq.attention_mass(cache, q, kc, corr=corr, flags=flags)
    torch.cuda.synchronize()
    assert kvq.last_device_status() == 0
    assert torch.allclose(ps2, ps, atol=1e-6) and torch.allclose(pr2, pr, atol=1e-6)
    assert torch.allclose(ps + pr, torch.ones_like(ps), atol=1e-5)


def test_split_workspace_and_small_workspace():
    """The workspace query covers the split partials (it exceeds the unsplit
    need); a workspace of only the unsplit size still gives the right answer
    (the launch falls back to one range)."""
    case = SPLIT[1]
    w, x, s, cache = _setup(case, seed=9)
    d, n_q, n_r, bh = case[0], case[3], case[5], case[8]
    up = lambda b: (b + 255) // 256 * 256
    # rotated query (high, low), rotated current values, two floats per head
    unsplit = 2 * up(bh * n_q * d * 2) + up(bh * n_r * d * 2) + 2 * up(bh * 4)
    assert cache.workspace_bytes(n_q, n_r) > unsplit
    q, kc, vc = x["q"].cuda(), x["k_cur"].cuda(), x["v_cur"].cuda()
    small = torch.empty(unsplit, dtype=torch.uint8, device="cuda")
    out, ps, pr = kvq.attention_corrected(cache, q, kc, vc, with_mass=True, workspace=small)
    torch.cuda.synchronize()
    assert kvq.last_device_status() == 0
    o_ref, ps_ref, pr_ref = oracle_head(w, x, s, 0, 0, np.arange(n_q), kvq.CORR_TAYLOR,
                                        n_s=case[4])
    assert_close(out[0, 0].float().cpu().numpy(), o_ref, ps[0, 0].cpu().numpy(), ps_ref,
                 pr[0, 0].cpu().numpy(), pr_ref, what="small workspace")
