"""Write the stored oracle answers that ``bench.py``'s accuracy report compares
the CUDA path with (``accuracy_w4.npz`` beside this script).

Calls only the oracle and the seeded input generator: for the INT2 g32 and
INT4 g64 four-chunk-window workloads (24 heads, head_dim 128, 4680-token
chunks, 18720-token window, the same seeds for both), on sampled heads and
query rows, it stores

* O, P_S and P_R of the corrected chunk attention over the quantized window
  for the three correction modes (none, the Taylor term, the exact term) --
  "Quantized Keys Steal Attention", Eq. (1) for the cache, the corrected score
  of the Fig. 3 caption, P_S and P_R as defined in section 1;
* P_S over the unquantized BF16 window (no quantization at all), the baseline
  of the attention-mass shift that the paper's abstract and Figure 2 describe;
* a SHA-256 fingerprint of each sampled head's BF16 inputs, so that a reader
  of the file can tell whether its own generator produced the same tensors.

Run from the repository root:  python tests/golden/make_accuracy_refs.py
(a minute or two on one core).
"""
from __future__ import annotations

import hashlib
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import kvq_oracle as O  # noqa: E402
from quantized_kv_cache_quantize_gb300 import synth  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "accuracy_w4.npz")
WORKLOADS = ("w4_int2", "w4_int4")
HEADS = (0, 23)
N_ROWS = 32
CORRS = (("none", O.CORR_NONE), ("taylor", O.CORR_TAYLOR), ("exact", O.CORR_EXACT))
INPUT_KEYS = ("q", "k_cur", "v_cur", "k_win", "v_win")


def sample_rows(n_q: int) -> np.ndarray:
    """The first and last query rows plus seeded ones in between."""
    rng = np.random.default_rng(1)
    mid = rng.choice(np.arange(1, n_q - 1), size=N_ROWS - 2, replace=False)
    return np.sort(np.concatenate([[0, n_q - 1], mid])).astype(np.int64)


def fingerprint(x: dict) -> str:
    """SHA-256 over the BF16 bit patterns of one head's inputs, in INPUT_KEYS order."""
    h = hashlib.sha256()
    for k in INPUT_KEYS:
        h.update(x[k].float().numpy().tobytes())   # BF16 -> fp32 is exact
    return h.hexdigest()


def head_refs(w: synth.Workload, h: int, rows: np.ndarray, signs: np.ndarray) -> dict:
    x = synth.head_inputs(w, h)
    kf = x["k_win"].float().numpy()
    vf = x["v_win"].float().numpy()
    kc_, vc_ = x["k_cur"].float().numpy(), x["v_cur"].float().numpy()
    q = x["q"].float().numpy()[rows]
    _, kd, kz, _, kc = O.quantize_rows(kf, signs, w.bits, w.group)
    _, vd, vz, _, vc = O.quantize_rows(vf, signs, w.bits, w.group)
    k_hat = O.dequantize(kc, kd, kz, w.group)
    v_hat = O.dequantize(vc, vd, vz, w.group)
    out = {"fp": fingerprint(x)}
    for name, corr in CORRS:
        o, ps, pr = O.chunk_attention(q, k_hat, v_hat, kd, kc_, vc_, signs, w.scale, w.group, corr)
        out[f"o_{name}"] = o.astype(np.float32)
        out[f"ps_{name}"] = ps
        out[f"pr_{name}"] = pr
    zero = np.zeros((kf.shape[0], w.head_dim // w.group))
    _, ps_u, _ = O.chunk_attention(q, O.rotate(kf, signs), O.rotate(vf, signs), zero, kc_, vc_,
                                   signs, w.scale, w.group, O.CORR_NONE)
    out["ps_unquantized"] = ps_u
    return out


def main() -> None:
    signs = synth.hadamard_signs(128)
    data = {}
    for name in WORKLOADS:
        w = synth.WORKLOADS[name]
        rows = sample_rows(w.n_q)
        data[f"{name}/heads"] = np.asarray(HEADS, dtype=np.int64)
        data[f"{name}/rows"] = rows
        per = [head_refs(w, h, rows, signs) for h in HEADS]
        for key in per[0]:
            vals = [p[key] for p in per]
            data[f"{name}/{key}"] = np.asarray(vals) if key != "fp" else np.asarray(vals, dtype="U64")
        print(f"{name}: heads {HEADS}, {len(rows)} rows", flush=True)
    np.savez_compressed(OUT, **data)
    print(f"wrote {OUT}")


if __name__ == "__main__":
    main()
