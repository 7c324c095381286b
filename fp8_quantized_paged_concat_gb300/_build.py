"""Builds libkvq.so, the sm_103a CUDA library behind include/kvq.h.

Each .cu file under csrc/ is compiled in parallel with nvcc for sm_103a only
(precise division and square root, no fast math: the quantizers rely on
IEEE-rounded divisions), then linked into
fp8_quantized_paged_concat_gb300/_lib/libkvq.so against the shared CUDA
runtime, the same one PyTorch loads.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(ROOT, "_build", "kvq")
LIBRARY = os.path.join(PKG, "_lib", "libkvq.so")

SOURCES = ["kvq_abi.cu", "kvq_write.cu", "kvq_gather.cu", "kvq_per_head.cu", "kvq_index.cu",
           "kvq_attention.cu", "kvq_selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-prec-div=true", "-prec-sqrt=true", "-ftz=false", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libkvq.so")
    return path


def _headers_mtime() -> float:
    paths = [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    paths += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, extra_flags=(), library: str = LIBRARY,
          objdir: str = OBJDIR) -> str:
    """Compiles and links libkvq.so if any source is newer; returns its path.
    ``extra_flags`` / ``library`` / ``objdir`` build a variant elsewhere (for
    example with -D tuning knobs) without touching the default library."""
    os.makedirs(objdir, exist_ok=True)
    os.makedirs(os.path.dirname(library), exist_ok=True)
    hdr = _headers_mtime()
    compiler = nvcc()

    def compile_one(src: str) -> str:
        s = os.path.join(CSRC, src)
        o = os.path.join(objdir, src.replace(".cu", ".o"))
        if force or not os.path.exists(o) or os.path.getmtime(o) < max(hdr, os.path.getmtime(s)):
            cmd = [compiler, *NVCC_FLAGS, *extra_flags, "-c", s, "-o", o]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
            if verbose and r.stderr:
                print(r.stderr)
        return o

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as pool:
        objs = list(pool.map(compile_one, SOURCES))
    if force or not os.path.exists(library) or os.path.getmtime(library) < max(map(os.path.getmtime, objs)):
        tmp = library + ".tmp.%d" % os.getpid()
        cmd = [compiler, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
               "-Xlinker", "-rpath," + os.path.join(os.path.dirname(os.path.dirname(compiler)), "lib64")]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"linking libkvq.so failed:\n{r.stderr}")
        os.replace(tmp, library)
    return library


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))
