"""The C ABI from a plain C program: tests/c/abi_example.c is compiled with
gcc against include/kvq.h, libkvq.so and the CUDA runtime (plus the oracle,
for the expected bytes) and run on the GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu


def test_c_program_uses_the_abi(tmp_path):
    from fp8_quantized_paged_concat_gb300 import _build
    from oracle import build as oracle_build
    lib = _build.build()
    oracle_build.build()
    cuda = os.path.dirname(os.path.dirname(_build.nvcc()))
    exe = str(tmp_path / "abi_example")
    cmd = [shutil.which("gcc") or "gcc", "-O2", "-std=c11", "-ffp-contract=off",
           os.path.join(ROOT, "tests", "c", "abi_example.c"), os.path.join(ROOT, "oracle", "kvq_oracle.c"),
           "-I" + os.path.join(ROOT, "include"), "-I" + os.path.join(ROOT, "oracle"),
           "-I" + os.path.join(cuda, "include"), "-L" + os.path.dirname(lib), "-lkvq",
           "-L" + os.path.join(cuda, "lib64"), "-lcudart", "-lm",
           "-Wl,-rpath," + os.path.dirname(lib) + ":" + os.path.join(cuda, "lib64"), "-o", exe]
    subprocess.run(cmd, check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bit for bit" in r.stdout
