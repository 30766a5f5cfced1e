"""Coefficients of the polynomial the exact-correction kernels use for
f(a) = log(sinh(a) / a) on 0 <= a <= 3 (the per-channel Jensen term of the
uniform rounding noise; "Quantized Keys Steal Attention", Fig. 3 caption).

With t = a^2, f = t h(t) where h is analytic on [0, 9] (its nearest
singularity is t = -pi^2).  h is interpolated at the N Chebyshev nodes of
[0, T_MAX] (a standard Chebyshev interpolation), and the interpolant is
rewritten in powers of t: f(a) ~ sum_{n=1..N} p_n t^n.  Being a polynomial in
a^2, the sum over a group's channels separates into the query's power sums
and the key's step size, as the kernels need; the fit extends the range of
that separation from a <= 1 (the Taylor series) to a <= 3.

Run: python quantized_kv_cache_quantize_gb300/csrc/sinhc_fit.py  (prints the
constants of kvq_attn_kernel.cuh's sinhc_fit).
"""
from __future__ import annotations

import numpy as np

T_MAX = 9.0
N_TERMS = 8


def h_of_t(t: np.ndarray) -> np.ndarray:
    """h(t) = log(sinh(sqrt t) / sqrt t) / t, with its series near 0."""
    t = np.asarray(t, dtype=np.float64)
    out = np.empty_like(t)
    small = t < 1e-3
    ts = t[small]
    out[small] = 1.0 / 6.0 - ts / 180.0 + ts * ts / 2835.0
    a = np.sqrt(t[~small])
    out[~small] = np.log(np.sinh(a) / a) / t[~small]
    return out


def fit_coefficients(n: int = N_TERMS, t_max: float = T_MAX) -> np.ndarray:
    """p_1 .. p_n (float64) of f(a) ~ sum p_k a^(2k) on a^2 in [0, t_max]."""
    from numpy.polynomial import chebyshev as C
    from numpy.polynomial import polynomial as P
    k = np.arange(n)
    x = np.cos(np.pi * (k + 0.5) / n)              # Chebyshev nodes on [-1, 1]
    c = C.chebfit(x, h_of_t((x + 1.0) * t_max / 2.0), n - 1)
    in_x = C.cheb2poly(c)                          # h as a polynomial in x
    in_t = np.zeros(1)
    for i, ci in enumerate(in_x):                  # x = 2 t / t_max - 1
        in_t = P.polyadd(in_t, ci * P.polypow([-1.0, 2.0 / t_max], i))
    return np.asarray(in_t[:n], dtype=np.float64)   # h = sum in_t[i] t^i, f = sum in_t[i] t^(i+1)


if __name__ == "__main__":
    for i, p in enumerate(fit_coefficients()):
        print(f"k == {i} ? {float(np.float32(p)):.9e}f")
