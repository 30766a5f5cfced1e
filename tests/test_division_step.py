"""The quantizer's exact-quotient step, checked on the CPU.

The CUDA quantizer gets fl(x / delta) for every element of a group from the
correctly rounded reciprocal and one FMA residual step instead of a division
per element.  Bit-exact codes (Eq. (1) with rint of the IEEE quotient) rest
on that identity, so it is swept here with IEEE float arithmetic in C (gcc,
no FMA contraction): every normal BF16 step size in a wide exponent range,
random numerators and every exact tie k + 1/2."""
import os
import shutil
import subprocess
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_division_step_matches_ieee_quotient():
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "division_step_check")
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-o", exe,
                               os.path.join(HERE, "division_step_check.c"), "-lm"])
        out = subprocess.run([exe, "-40", "20", "2000"], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "mismatches 0" in out.stdout


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_row_divisor_matches_integer_division():
    """The quantize-append kernels find a row's (batch, head) as r / n_new by
    a multiply-high and a shift (the host picks both once per call); the
    quotient must equal the integer division for every row index below 2^31
    (the host refuses larger launches)."""
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "row_divisor_check")
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-I", cuda_inc, "-o", exe,
                               os.path.join(HERE, "row_divisor_check.cpp")])
        out = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "bad 0" in out.stdout
