"""The exact correction's power series, checked on the CPU.

The GPU evaluates log(sinh a / a) = sum_k c_k a^(2k) through k = 7 (the
coefficients are constants of the attention kernel header).  Here a host
program built from that header with nvcc prints them, and they are compared
with c_k = 2^(2k) B_2k / (2k (2k)!) (B the Bernoulli numbers) and with the
oracle's log_sinhc: the truncated series must meet it within the bound the
kernels rely on (|c_8| a^16 per channel for a <= 1)."""
import fractions
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

from oracle import kvq_oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))


def _coef(k: int) -> fractions.Fraction:
    sympy = pytest.importorskip("sympy")
    b = sympy.bernoulli(2 * k)
    return fractions.Fraction(2 ** (2 * k)) * fractions.Fraction(int(b.p), int(b.q)) / (
        2 * k * fractions.Fraction(int(sympy.factorial(2 * k))))


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


@pytest.mark.skipif(_nvcc() is None, reason="needs nvcc")
def test_kernel_series_coefficients():
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "series_coef_check")
        subprocess.check_call([_nvcc(), "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
                               "-o", exe, os.path.join(HERE, "series_coef_check.cu")])
        out = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    vals = out.stdout.split()
    n = int(vals[0])
    got = [float(v) for v in vals[1:]]
    assert n == len(got) == 7
    for k, g in enumerate(got, start=1):
        want = float(_coef(k))
        assert abs(g - want) <= 2 ** -23 * abs(want), (k, g, want)
    # the truncated series against the oracle's log(sinh a / a) on a <= 1
    a = np.linspace(0.0, 1.0, 1001)
    t = a * a
    series = sum(float(_coef(k)) * t ** k for k in range(1, n + 1))
    bound = abs(float(_coef(n + 1))) * t ** (n + 1) * 1.01 + 1e-16
    assert np.all(np.abs(series - O.log_sinhc(a)) <= bound)
