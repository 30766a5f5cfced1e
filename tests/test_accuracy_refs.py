"""The stored oracle answers of the accuracy report (tests/golden/accuracy_w4.npz)
are the oracle's: recomputed here for a few of the stored rows."""
from __future__ import annotations

import os

import numpy as np

from oracle import kvq_oracle as O
from quantized_kv_cache_quantize_gb300 import synth
from tests.golden import make_accuracy_refs as M

NPZ = os.path.join(os.path.dirname(__file__), "golden", "accuracy_w4.npz")


def test_stored_refs_match_the_oracle():
    z = np.load(NPZ)
    w = synth.WORKLOADS["w4_int4"]
    heads = z["w4_int4/heads"]
    rows = z["w4_int4/rows"]
    assert list(heads) == list(M.HEADS) and np.array_equal(rows, M.sample_rows(w.n_q))
    h = int(heads[1])
    pick = [0, 7, len(rows) - 1]
    x = synth.head_inputs(w, h)
    assert M.fingerprint(x) == str(z["w4_int4/fp"][1])
    signs = synth.hadamard_signs(128)
    kf = x["k_win"].float().numpy()
    vf = x["v_win"].float().numpy()
    _, kd, kz, _, kc = O.quantize_rows(kf, signs, w.bits, w.group)
    _, vd, vz, _, vc = O.quantize_rows(vf, signs, w.bits, w.group)
    q = x["q"].float().numpy()[rows[pick]]
    o, ps, pr = O.chunk_attention(q, O.dequantize(kc, kd, kz, w.group), O.dequantize(vc, vd, vz, w.group),
                                  kd, x["k_cur"].float().numpy(), x["v_cur"].float().numpy(), signs,
                                  w.scale, w.group, O.CORR_TAYLOR)
    np.testing.assert_allclose(o.astype(np.float32), z["w4_int4/o_taylor"][1][pick], rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(ps, z["w4_int4/ps_taylor"][1][pick], rtol=0, atol=1e-12)
    np.testing.assert_allclose(pr, z["w4_int4/pr_taylor"][1][pick], rtol=0, atol=1e-12)
    # the mass identity P_S + P_R = 1 on every stored row and mode
    for name in ("w4_int2", "w4_int4"):
        for c in ("none", "taylor", "exact"):
            np.testing.assert_allclose(z[f"{name}/ps_{c}"] + z[f"{name}/pr_{c}"], 1.0, atol=1e-12)
