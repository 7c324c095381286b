"""The fp8_ds_mla write kernel's division-free arithmetic against IEEE
division: the quotient x / s (Markstein's correction after a correctly
rounded reciprocal, tile scales below 2^-64 rescaled by 2^96) for every pair
of bf16 values x, amax with |x| <= amax -- the e4m3 code it feeds is the
oracle's -- and the stored tile scale amax / 448 for every bf16 amax.  Host
code only (tests/c/fp8_quotient_check.c); a few seconds on several cores (about half a minute on one)."""
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
def test_fp8_quotient_matches_ieee_division_exhaustively(tmp_path):
    exe = tmp_path / "fp8_quotient_check"
    openmp = ["-fopenmp"] if _has_openmp(tmp_path) else []
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", *openmp, "-o", str(exe),
                           os.path.join(HERE, "c", "fp8_quotient_check.c"), "-lm"])
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout
    assert "pairs 1065402238 mismatches 0" in r.stdout
    assert "scales 32639 scale mismatches 0" in r.stdout
