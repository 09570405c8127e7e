"""The E4M3 row quantiser divides by the row scale with one reciprocal per row
and Markstein's correction step per value. That the step reproduces the
correctly rounded quotient over the quantiser's whole input domain (scales in
its fast range) is checked here exhaustively on the CPU, in IEEE fp32 with
fused multiply-adds (quantize_division_check.c)."""
import os
import shutil
import subprocess
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_reciprocal_correction_step_is_the_correctly_rounded_quotient():
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "check")
        subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-o", exe,
                        os.path.join(HERE, "quantize_division_check.c"), "-lm"], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stdout + out.stderr
    rows, pairs, bad = (int(t) for t in out.stdout.split()[1::2])
    assert bad == 0 and rows == 28064 and pairs > 10 ** 9, out.stdout
