"""The write kernels' division-free NVFP4 group scale (Markstein's correction
of amax * RN(1/6)) against IEEE division, for every non-negative fp32 amax:
the e4m3 scale code is the oracle's.  Host code only
(tests/c/nvfp4_scale_check.c); about half a minute on one core."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_nvfp4_scale_matches_ieee_division_exhaustively(tmp_path):
    exe = tmp_path / "nvfp4_scale_check"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-o", str(exe),
                           os.path.join(HERE, "c", "nvfp4_scale_check.c"), "-lm"])
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout
    assert "mismatches 0" in r.stdout
    assert "values 2139095041" in r.stdout
