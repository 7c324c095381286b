"""The write kernels' division-free NVFP4 group scale (Markstein's correction
of amax * RN(1/6)) against IEEE division, for every non-negative fp32 amax:
the e4m3 scale code is the oracle's.  Host code only
(tests/c/nvfp4_scale_check.c); a few seconds on several cores (about half a minute on one)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def _has_openmp(tmp_path):
    """Whether gcc links OpenMP here (the check then uses every core)."""
    src = tmp_path / "omp.c"
    src.write_text("int main(void) { return 0; }\n")
    return subprocess.run(["gcc", "-fopenmp", "-o", str(tmp_path / "omp"), str(src)],
                          capture_output=True).returncode == 0


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_nvfp4_scale_matches_ieee_division_exhaustively(tmp_path):
    exe = tmp_path / "nvfp4_scale_check"
    openmp = ["-fopenmp"] if _has_openmp(tmp_path) else []
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", *openmp, "-o", str(exe),
                           os.path.join(HERE, "c", "nvfp4_scale_check.c"), "-lm"])
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout
    assert "mismatches 0" in r.stdout
    assert "values 2139095041" in r.stdout
