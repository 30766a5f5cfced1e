"""Seeded synthetic inputs for the chunk-attention workloads.

This module only draws random numbers and casts them to BF16. It holds none of
the method's arithmetic (no rotation, no quantization, no attention), so that
both the CUDA path and the CPU oracle can consume the very same inputs.

Workloads are "video-shaped": token counts are latent frames x height x width
of a chunk-wise autoregressive video diffusion model (the paper evaluates on
MAGI-1, SkyReels-V2 and HY-WorldPlay; none of their weights or prompts is used
here, the tensors below stand in for the attention inputs of one layer).

Distributions (per head h, generator ``numpy.random.default_rng((seed, h))``):

* queries and values: N(0, 1);
* keys: N(0, 1) (or Student-t(3) per channel for the high-resolution case),
  optionally plus a per-channel mean offset mu_c ~ N(0, offset_std^2), with a
  few distinct "outlier" channels multiplied by ``outlier_scale`` -- keys in
  transformers show channel-wise outliers (Quantized Keys Steal Attention,
  section 3 "Hadamard rotation").

Draw order per head: Q, K_cur, V_cur, K_window, V_window, K_new, V_new, then
the outlier channels (distinct, chosen before rotation) and the offsets.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    heads: int
    head_dim: int
    chunk_tokens: int          # current-chunk length N_R (= number of queries N_q)
    n_chunks: int              # cache window in chunks; N_S = chunk_tokens * n_chunks
    bits: int
    group: int
    key_dist: str = "normal"   # "normal" or "t3"
    outlier_frac: float = 0.0  # fraction of channels that are outliers (ceil)
    n_outliers_fixed: int = 0  # used instead of outlier_frac when > 0
    outlier_scale: float = 1.0
    offset_std: float = 0.0
    batch: int = 1

    @property
    def n_q(self) -> int:
        return self.chunk_tokens

    @property
    def n_r(self) -> int:
        return self.chunk_tokens

    @property
    def n_s(self) -> int:
        return self.chunk_tokens * self.n_chunks

    @property
    def n_outliers(self) -> int:
        if self.n_outliers_fixed > 0:
            return self.n_outliers_fixed
        return int(math.ceil(self.outlier_frac * self.head_dim - 1e-9))

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def attention_flops(self, n_q=None, n_s=None, n_r=None, heads=None) -> float:
        """Algorithmic FLOPs of one corrected chunk attention: QK^T and PV over
        both segments, plus the bias term (2 flops per cached score and group)."""
        n_q = self.n_q if n_q is None else n_q
        n_s = self.n_s if n_s is None else n_s
        n_r = self.n_r if n_r is None else n_r
        bh = self.batch * (self.heads if heads is None else heads)
        d = self.head_dim
        g = d // self.group
        return 4.0 * n_q * (n_s + n_r) * d * bh + 2.0 * n_q * n_s * g * bh

    def append_bytes(self, n_new: int | None = None) -> float:
        """Algorithmic HBM bytes of one quantize-append of ``n_new`` tokens:
        read BF16 K and V, write packed codes and the BF16 (step, zero) pairs."""
        n = self.chunk_tokens if n_new is None else n_new
        bh = self.batch * self.heads
        d = self.head_dim
        g = d // self.group
        per_row = d * 2 + d * self.bits // 8 + g * 2 * 2
        return float(2 * n * bh * per_row)


WORKLOADS = {
    # 1 head, d 64, 256-token chunk over a 1024-token INT2 g32 window.
    "tiny": Workload("tiny", heads=1, head_dim=64, chunk_tokens=256, n_chunks=4,
                     bits=2, group=32, n_outliers_fixed=4, outlier_scale=8.0),
    # One layer, 24 heads, 3 latent frames x 30 x 52 per chunk, 4-chunk window.
    "w4_int2": Workload("w4_int2", heads=24, head_dim=128, chunk_tokens=4680,
                        n_chunks=4, bits=2, group=32, outlier_frac=0.02,
                        outlier_scale=10.0, offset_std=0.5),
    # Same shapes and seeds, INT4 with groups of 64.
    "w4_int4": Workload("w4_int4", heads=24, head_dim=128, chunk_tokens=4680,
                        n_chunks=4, bits=4, group=64, outlier_frac=0.02,
                        outlier_scale=10.0, offset_std=0.5),
    # Long window: 32 heads, 4 latent frames x 30 x 52, 8-chunk window.
    "w8_int2": Workload("w8_int2", heads=32, head_dim=128, chunk_tokens=6240,
                        n_chunks=8, bits=2, group=32, outlier_frac=0.02,
                        outlier_scale=10.0, offset_std=0.5),
    # High-resolution streaming step: 40 heads, 4 x 60 x 60, 6-chunk window,
    # Student-t(3) keys with 1% outlier channels at 12x.
    "hires_t3": Workload("hires_t3", heads=40, head_dim=128, chunk_tokens=14400,
                         n_chunks=6, bits=2, group=32, key_dist="t3",
                         outlier_frac=0.01, outlier_scale=12.0),
}


def with_sizes(w: Workload, **kw) -> Workload:
    """A copy of a workload with some fields changed (used for ragged tests)."""
    return replace(w, **kw)


def _keys(rng, n, d, w: Workload) -> np.ndarray:
    if w.key_dist == "t3":
        return rng.standard_t(3, size=(n, d)).astype(np.float32)
    return rng.standard_normal((n, d), dtype=np.float32)


def _to_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def head_inputs(w: Workload, head: int, seed: int = 0, n_q: int | None = None,
                n_s: int | None = None, n_r: int | None = None,
                n_new: int | None = None) -> dict:
    """BF16 tensors of one (batch 0) head: q [n_q,d], k_cur/v_cur [n_r,d],
    k_win/v_win [n_s,d] (the window to be quantized), k_new/v_new [n_new,d]."""
    d = w.head_dim
    n_q = w.n_q if n_q is None else n_q
    n_s = w.n_s if n_s is None else n_s
    n_r = w.n_r if n_r is None else n_r
    n_new = w.chunk_tokens if n_new is None else n_new
    rng = np.random.default_rng((seed, head))
    q = rng.standard_normal((n_q, d), dtype=np.float32)
    k_cur = _keys(rng, n_r, d, w)
    v_cur = rng.standard_normal((n_r, d), dtype=np.float32)
    k_win = _keys(rng, n_s, d, w)
    v_win = rng.standard_normal((n_s, d), dtype=np.float32)
    k_new = _keys(rng, n_new, d, w)
    v_new = rng.standard_normal((n_new, d), dtype=np.float32)
    n_out = w.n_outliers
    if n_out > 0:
        chans = rng.choice(d, size=n_out, replace=False)
        for k in (k_cur, k_win, k_new):
            k[:, chans] *= np.float32(w.outlier_scale)
    if w.offset_std > 0:
        mu = (rng.standard_normal(d) * w.offset_std).astype(np.float32)
        for k in (k_cur, k_win, k_new):
            k += mu
    return {"q": _to_bf16(q), "k_cur": _to_bf16(k_cur), "v_cur": _to_bf16(v_cur),
            "k_win": _to_bf16(k_win), "v_win": _to_bf16(v_win),
            "k_new": _to_bf16(k_new), "v_new": _to_bf16(v_new)}


def inputs(w: Workload, seed: int = 0, heads=None, **sizes) -> dict:
    """Stacked BF16 tensors [1, H, N, d] for the given heads (default: all)."""
    hs = range(w.heads) if heads is None else heads
    per = [head_inputs(w, h, seed, **sizes) for h in hs]
    return {k: torch.stack([p[k] for p in per])[None].contiguous() for k in per[0]}


def hadamard_signs(d: int, seed: int = 0) -> np.ndarray:
    """Random +-1 diagonal of the randomized Hadamard rotation (float32)."""
    rng = np.random.default_rng((seed, 0x5167))
    return np.where(rng.integers(0, 2, size=d) == 1, -1.0, 1.0).astype(np.float32)
