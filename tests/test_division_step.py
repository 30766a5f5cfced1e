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
