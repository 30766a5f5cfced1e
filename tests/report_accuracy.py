"""Accuracy report over the workloads: the CUDA path against the oracle, and the
shift of attention mass onto the quantized cache with and without the Jensen
correction ("Quantized Keys Steal Attention", abstract and Figure 2: quantized
keys take attention mass from the current chunk; the correction gives it
back).  INT4 g64 and INT2 g32 run on the same seeds.

Run on a GPU:  python tests/report_accuracy.py [--heads 3] [--rows 512]
               [--corrs none,taylor,exact] [--keys token|channel]

For every workload, sampled heads and query rows:
  err_O   max |O_gpu - O_oracle| / max |O_oracle|           (same quantized cache)
  err_PS  max |P_S_gpu - P_S_oracle|
  P_S     mean mass on the cache: GPU, oracle with the quantized cache, and
          oracle with the unquantized BF16 cache (no quantization at all);
          shift = P_S(quantized) - P_S(unquantized), per correction mode.
Prints one table; the oracle inputs are the seeded BF16 tensors only.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import kvq_oracle as O  # noqa: E402
from quantized_kv_cache_quantize_gb300 import kvq, synth  # noqa: E402
from tests.gpu_common import (build_cache, build_cache_kch, oracle_head,  # noqa: E402
                              oracle_head_kch)

CORRS = {"none": kvq.CORR_NONE, "taylor": kvq.CORR_TAYLOR, "exact": kvq.CORR_EXACT}


def unquantized_head(w, x, signs, h, rows):
    """Oracle attention over the exact BF16 window (no quantization)."""
    kf = x["k_win"][0, h].float().numpy()
    vf = x["v_win"][0, h].float().numpy()
    q = x["q"][0, h].float().numpy()[rows]
    zero = np.zeros((kf.shape[0], w.head_dim // w.group))
    return O.chunk_attention(q, O.rotate(kf, signs), O.rotate(vf, signs), zero,
                             x["k_cur"][0, h].float().numpy(), x["v_cur"][0, h].float().numpy(),
                             signs, w.scale, w.group, O.CORR_NONE)


def report(name, n_heads, n_rows, flags, corrs, keys):
    w = synth.WORKLOADS[name]
    x = synth.inputs(w)
    s = synth.hadamard_signs(w.head_dim)
    channel = keys == "channel"
    cache = (build_cache_kch if channel else build_cache)(w, x, s)
    ref_head = oracle_head_kch if channel else oracle_head
    q, kc, vc = x["q"].cuda(), x["k_cur"].cuda(), x["v_cur"].cuda()
    gpu = {}
    for corr in corrs:
        out, ps, pr = kvq.attention_corrected(cache, q, kc, vc, corr=corr, with_mass=True, flags=flags)
        torch.cuda.synchronize()
        assert kvq.last_device_status() == 0
        gpu[corr] = (out.float().cpu().numpy(), ps.cpu().numpy())
    rng = np.random.default_rng(1)
    heads = np.linspace(0, w.heads - 1, n_heads).astype(int)
    rows = np.sort(rng.choice(w.n_q, size=min(n_rows, w.n_q), replace=False))
    lines = []
    acc = {c: {"err_o": 0.0, "err_ps": 0.0, "ps_gpu": [], "ps_ora": []} for c in gpu}
    ps_exact = []
    for h in heads:
        _, ps_u, _ = unquantized_head(w, x, s, h, rows)
        ps_exact.append(ps_u)
        for corr in gpu:
            o_ref, ps_ref, _ = ref_head(w, x, s, 0, h, rows, corr)
            o_g, ps_g = gpu[corr][0][0, h][rows], gpu[corr][1][0, h][rows]
            a = acc[corr]
            a["err_o"] = max(a["err_o"], float(np.abs(o_g - o_ref).max() / np.abs(o_ref).max()))
            a["err_ps"] = max(a["err_ps"], float(np.abs(ps_g - ps_ref).max()))
            a["ps_gpu"].append(ps_g)
            a["ps_ora"].append(ps_ref)
    p_exact = float(np.mean(np.concatenate(ps_exact)))
    for corr, a in acc.items():
        p_gpu = float(np.mean(np.concatenate(a["ps_gpu"])))
        p_ora = float(np.mean(np.concatenate(a["ps_ora"])))
        cname = {v: k for k, v in CORRS.items()}[corr]
        lines.append(f"| {name} | INT{w.bits} g{w.group} {keys} | {cname} | "
                     f"{a['err_o']:.2e} | {a['err_ps']:.2e} | {p_gpu:.5f} | {p_ora:.5f} | "
                     f"{p_exact:.5f} | {p_gpu - p_exact:+.5f} |")
    return lines


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--heads", type=int, default=3)
    ap.add_argument("--rows", type=int, default=512)
    ap.add_argument("--workloads", default="w4_int2,w4_int4,w8_int2,hires_t3")
    ap.add_argument("--corrs", default="none,taylor",
                    help="comma-separated: none, taylor, exact (the oracle's exact term "
                         "is slow on long windows: fewer rows)")
    ap.add_argument("--keys", choices=["token", "channel"], default="token")
    args = ap.parse_args(argv)
    corrs = [CORRS[c] for c in args.corrs.split(",")]
    print(f"sampled heads per workload: {args.heads}, query rows per head: {args.rows}")
    print("| workload | cache | correction | err_O | err_PS | P_S gpu | P_S oracle | "
          "P_S unquantized | shift (gpu - unquantized) |")
    print("|---|---|---|---|---|---|---|---|---|")
    for name in args.workloads.split(","):
        flags = kvq.FLAG_PRECISE_QUERY if name == "hires_t3" else 0
        for line in report(name, args.heads, args.rows, flags, corrs, args.keys):
            print(line, flush=True)


if __name__ == "__main__":
    main()
