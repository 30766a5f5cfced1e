"""The checked build (libkvq_checked.so: the same sources with
-DKVQ_DEBUG_BOUNDS, every kernel testing the indices of its global-memory
accesses) runs the parity cases without a failed check: quantize-append of
ragged chunks per token and per channel, the rotation, the attention in every
correction mode with and without the key-range split and the staged words,
and the SM-pair kernel; results still match the oracle.  It runs in a child
process, which loads the checked library through KVQ_LIBRARY."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import numpy as np, torch
from oracle import kvq_oracle as O
from quantized_kv_cache_quantize_gb300 import kvq, synth
from tests.gpu_common import build_cache, build_cache_kch, oracle_head, oracle_head_kch, assert_close

assert kvq.debug_bounds_build()

def clean(what):
    torch.cuda.synchronize()
    st, site = kvq.last_device_status(), kvq.debug_bounds_site()
    assert st == 0 and site == 0, (what, st, site)

cases = [  # d, bits, group, n_q, n_s, n_r, chunk, n_chunks, heads, key mode
    (128, 2, 32, 300, 1000, 129, 300, 4, 2, kvq.KEYS_PER_TOKEN),
    (128, 4, 64, 129, 257, 64, 128, 3, 1, kvq.KEYS_PER_TOKEN),
    (64, 2, 32, 200, 390, 77, 100, 4, 2, kvq.KEYS_PER_TOKEN),
    (128, 2, 32, 150, 700, 60, 300, 3, 2, kvq.KEYS_PER_CHANNEL),
]
for d, bits, group, n_q, n_s, n_r, chunk, n_chunks, heads, km in cases:
    w = synth.Workload("checked", heads=heads, head_dim=d, chunk_tokens=chunk, n_chunks=n_chunks,
                       bits=bits, group=group, n_outliers_fixed=2, outlier_scale=6.0)
    x = synth.inputs(w, seed=3, n_q=n_q, n_s=n_s, n_r=n_r)
    s = synth.hadamard_signs(d, seed=5)
    cache = (build_cache_kch if km == kvq.KEYS_PER_CHANNEL else build_cache)(w, x, s)
    clean(("append", d, bits, km))
    ref_head = oracle_head_kch if km == kvq.KEYS_PER_CHANNEL else oracle_head
    flag_sets = [0, kvq.FLAG_NO_KV_SPLIT, kvq.FLAG_PRECISE_QUERY, kvq.FLAG_STAGED_WORDS]
    for corr in (kvq.CORR_TAYLOR, kvq.CORR_NONE, kvq.CORR_EXACT):
        for flags in flag_sets:
            out, ps, pr = kvq.attention_corrected(cache, x["q"].cuda(), x["k_cur"].cuda(),
                                                  x["v_cur"].cuda(), corr=corr, with_mass=True,
                                                  flags=flags)
            clean(("attention", d, bits, km, corr, flags))
        rows = np.array([0, n_q // 2, n_q - 1])
        for h in range(heads):
            o_ref, ps_ref, pr_ref = ref_head(w, x, s, 0, h, rows, corr)
            assert_close(out[0, h, rows].float().cpu().numpy(), o_ref, ps[0, h, rows].cpu().numpy(),
                         ps_ref, pr[0, h, rows].cpu().numpy(), pr_ref, what=f"checked {d} {corr}")
    ms, mr = kvq.attention_mass(cache, x["q"].cuda(), x["k_cur"].cuda())
    clean(("mass", d, bits, km))
xr = synth.inputs(synth.WORKLOADS["tiny"], seed=1, n_q=300)["q"].cuda()
kvq.rotate(xr, synth.hadamard_signs(64))
kvq.rotate(xr, synth.hadamard_signs(64), torch.float16)
clean("rotate")
print("checked build clean")
'''


def test_checked_build_runs_clean():
    sys.path.insert(0, ROOT)
    from quantized_kv_cache_quantize_gb300 import build as b
    lib = b.build(checked=True)
    env = dict(os.environ, KVQ_LIBRARY=lib, PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "checked build clean" in r.stdout
