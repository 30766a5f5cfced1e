"""The allocation-free attention entry point against the ordinary one and the
oracle.

kvq_attention_corrected_noalloc serves callers that cannot allocate device
memory when they call (its scratch is a fixed buffer inside the library).
Through the C ABI, two calls in a row -- different problem sizes, so the
second one runs over whatever the first left in the shared buffer -- must
give what kvq_attention_corrected gives with a caller-allocated workspace,
within the tolerances of the other attention tests, and what the CPU oracle
gives for every row of one head.  Collected last, so a run that stops at its
first failure has run everything else already."""
import numpy as np
import pytest
import torch

from quantized_kv_cache_quantize_gb300 import kvq, synth
from tests.gpu_common import MASS_TOL, O_TOL, assert_close, build_cache, oracle_head

pytestmark = pytest.mark.gpu


def _case(name, heads, d, chunk, n_chunks, n_q, n_s, n_r, seed):
    w = synth.Workload(name, heads=heads, head_dim=d, chunk_tokens=chunk, n_chunks=n_chunks,
                       bits=2, group=32, n_outliers_fixed=3, outlier_scale=8.0, offset_std=0.4)
    x = synth.inputs(w, seed=seed, n_q=n_q, n_s=n_s, n_r=n_r)
    s = synth.hadamard_signs(d, seed=seed)
    cache = build_cache(w, x, s, n_s=n_s)
    return cache, {k: v.cuda() for k, v in x.items()}, (w, x, s)


def _compare(cache, x, host, flags):
    ref_o, ref_ps, ref_pr = kvq.attention_corrected(cache, x["q"], x["k_cur"], x["v_cur"],
                                                    with_mass=True, flags=flags)
    o, ps, pr = kvq.attention_corrected_noalloc(cache, x["q"], x["k_cur"], x["v_cur"],
                                                with_mass=True, flags=flags)
    torch.cuda.synchronize()
    assert kvq.last_device_status() == kvq.KVQ_OK
    ref = ref_o.float()
    err = (o.float() - ref).abs().max().item()
    assert err <= O_TOL * ref.abs().max().item()
    assert (ps - ref_ps).abs().max().item() <= MASS_TOL
    assert (pr - ref_pr).abs().max().item() <= MASS_TOL
    # and the oracle, from the same seeded inputs, on every row of head 0
    w, xh, s = host
    rows = np.arange(xh["q"].shape[2])
    o_ref, ps_ref, pr_ref = oracle_head(w, xh, s, 0, 0, rows, kvq.CORR_TAYLOR)
    assert_close(o[0, 0].float().cpu().numpy(), o_ref, ps[0, 0].cpu().numpy(), ps_ref,
                 pr[0, 0].cpu().numpy(), pr_ref, what="noalloc vs oracle")


def test_noalloc_matches_workspace_entry_point_twice():
    first = _case("a", heads=3, d=128, chunk=300, n_chunks=3, n_q=450, n_s=900, n_r=300, seed=21)
    second = _case("b", heads=2, d=64, chunk=128, n_chunks=2, n_q=129, n_s=200, n_r=77, seed=22)
    assert first[0].workspace_bytes(450, 300) <= kvq.NOALLOC_SCRATCH_BYTES
    _compare(*first, flags=0)
    _compare(*second, flags=kvq.FLAG_PRECISE_QUERY)
