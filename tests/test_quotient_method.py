"""The vector quantizers form w / s with Markstein's correction instead of an
IEEE division (csrc/quantize.cu).  This host-side check runs the same
binary32 steps over the whole domain they are used on -- every bf16 amax with
s = amax / 448 >= 2^-92 and every bf16 |w| <= amax, about 1.03e9 pairs --
and requires the e4m3 code of every quotient to equal the code of the IEEE
quotient.  (The GPU parity tests then compare the kernels' codes with the
oracle, which divides.)"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
def test_markstein_quotient_encodes_like_ieee_division(tmp_path):
    exe = tmp_path / "quotient_method"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
                    "-o", str(exe), os.path.join(HERE, "csrc", "quotient_method.c"), "-lm"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True, timeout=600).stdout.split()
    pairs, mismatches = int(out[1]), int(out[3])
    assert pairs > 1_000_000_000
    assert mismatches == 0
