"""Failure detection of the sparse MLA attention kernel on the GPU: its
bounded waits run out and the kernel reports it.

The kernel waits only through mbarriers, each wait with an iteration limit.
A build of the library used only here (KVQ_ATTN_STALL_TILE) makes the MMA
thread stop issuing at tile 2 of 4, as if its tensor work never completed, and
shortens the role waits' limit (KVQ_ATTN_WAIT_CYCLES, about 10 ms) so that
the test is quick; the final wait (for the CTA's own MMAs in flight) keeps its
own long limit.  Nothing hangs: the waits that nothing will satisfy run out,
every role takes the abort path, the kernel drains the MMAs it issued, frees
its tensor memory and returns.

Checked, in a process of its own: the call returns, KVQ_STATUS_TIMEOUT is set,
the outputs (out and lse) are untouched, and the normal library then gives a
correct result on the same device in the same process (against the oracle,
within the bound of tests/test_gpu_attention.py).
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
STALL_FLAGS = ["-DKVQ_ATTN_STALL_TILE=2", "-DKVQ_ATTN_WAIT_CYCLES=20000000LL"]


@pytest.fixture(scope="module")
def stall_library():
    from fp8_quantized_paged_concat_gb300 import _build
    _build.build()
    return _build.build(extra_flags=STALL_FLAGS, library=os.path.join(_build.PKG, "_lib", "libkvq_stall.so"),
                        objdir=os.path.join(_build.ROOT, "_build", "kvq_stall"))


def test_attention_waits_time_out_and_report(stall_library, oracle_mod, tmp_path):
    from test_gpu_attention import check, host_cache

    # 2 tokens x 16 heads, top-256 (four 64-slot tiles), 10 % unused slots
    w = wl.make_attention("timeout", 2, 16, 256, 8, 64, 351, p_unused=0.1)
    cache = host_cache(oracle_mod, w.fill)
    np.save(tmp_path / "q.npy", wl.bf16_bits(w.q))
    np.save(tmp_path / "indices.npy", wl.host(w.indices))
    np.save(tmp_path / "cache.npy", cache)
    np.save(tmp_path / "scale.npy", np.float64(w.softmax_scale))
    r = subprocess.run([sys.executable, os.path.join(HERE, "attention_timeout_child.py"), stall_library,
                        str(tmp_path)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    rep = json.loads(r.stdout.strip().splitlines()[-1])
    assert rep["rc"] == 0, rep
    assert rep["status"] & 0x4, f"KVQ_STATUS_TIMEOUT not set: {rep}"
    assert rep["out_untouched"] and rep["lse_untouched"], f"an aborted token wrote outputs: {rep}"
    assert rep["normal_status"] == 0, rep
    out = torch.from_numpy(np.load(tmp_path / "out.npy")).to(torch.bfloat16)
    lse = torch.from_numpy(np.load(tmp_path / "lse.npy"))
    check(oracle_mod, cache, w.q, wl.host(w.indices), w.softmax_scale, out, lse)
