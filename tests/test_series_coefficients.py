"""The exact correction's polynomial, checked on the CPU.

The GPU evaluates log(sinh a / a) as sum_k p_k a^(2k) through k = 8 for
a <= 3: over a group's channels through the query's power sums and the key's
step (the separable form), and per channel where a group leaves that range.
The p_k are a Chebyshev fit (derived by sinhc_fit.py beside the kernel
header).  A host program built from the header with nvcc prints them; they
must equal the generator's, rounded to fp32, and the polynomial evaluated in
fp32 the way the kernels do must meet the oracle's log_sinhc within 5e-7 on
0 <= a <= 3.  The first coefficients must also approach the Taylor series'
c_k = 2^(2k) B_2k / (2k (2k)!) (B the Bernoulli numbers), which the fit
reproduces near a = 0."""
import fractions
import importlib.util
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

from oracle import kvq_oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))


def _taylor(k: int) -> fractions.Fraction:
    sympy = pytest.importorskip("sympy")
    b = sympy.bernoulli(2 * k)
    return fractions.Fraction(2 ** (2 * k)) * fractions.Fraction(int(b.p), int(b.q)) / (
        2 * k * fractions.Fraction(int(sympy.factorial(2 * k))))


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


def _generator():
    path = os.path.join(HERE, "..", "quantized_kv_cache_quantize_gb300", "csrc", "sinhc_fit.py")
    spec = importlib.util.spec_from_file_location("sinhc_fit", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.skipif(_nvcc() is None, reason="needs nvcc")
def test_kernel_fit_coefficients():
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "series_coef_check")
        subprocess.check_call([_nvcc(), "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
                               "-I", os.path.join(HERE, "..", "include"),
                               "-o", exe, os.path.join(HERE, "series_coef_check.cu")])
        out = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    vals = out.stdout.split()
    nf, t_max = int(vals[0]), float(vals[1])
    fit = np.array([float(v) for v in vals[2:2 + nf]])
    assert len(fit) == nf
    mod = _generator()
    assert (nf, t_max) == (mod.N_TERMS, mod.T_MAX) == (8, 9.0)
    # the header's constants are the generator's, rounded to fp32 (printed
    # with 10 significant digits, which round-trip fp32)
    np.testing.assert_array_equal(fit.astype(np.float32), mod.fit_coefficients().astype(np.float32))
    # fp32 Horner in t = a^2, as the kernels evaluate it, against the oracle
    a = np.linspace(0.0, np.sqrt(t_max), 4001)
    t = (a * a).astype(np.float32)
    acc = np.full_like(t, np.float32(fit[-1]))
    for c in fit[-2::-1]:
        acc = (acc * t + np.float32(c)).astype(np.float32)
    err = np.abs((acc * t).astype(np.float64) - O.log_sinhc(a))
    assert err.max() <= 5e-7, err.max()
    # near 0 the fit is the Taylor series: c_1 = 1/6, c_2 = -1/180
    for k in (1, 2):
        want = float(_taylor(k))
        assert abs(fit[k - 1] - want) <= 1e-3 * abs(want), (k, fit[k - 1], want)
