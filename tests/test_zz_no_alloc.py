"""The split-key decode without a caller workspace
(kvq_sparse_mla_attention_split_nvfp4_ds_mla_noalloc).

Callers that cannot allocate device memory when they call in -- an engine
that reserved the GPU's memory for its own pools at start-up, or host code on
a latency-critical path where an allocation can synchronise the device --
use this entry point: its partial results go to a fixed array the library
holds on every GPU that loads it.  Checked here, through the C ABI (the
ctypes binding), on two calls in a row with different inputs (the second
call reuses the array the first one left behind): each output equals, bit
for bit, what kvq_sparse_mla_attention_split_nvfp4_ds_mla computes with a
workspace and the same number of key ranges, and lies within the error bound
the other attention tests use against the oracle.  A call that needs more
than the array holds is refused before anything is launched.

This file is collected last, so that a run stopping at its first failure has
run every other test before this one; it passes alone in a fresh process as
well.
"""
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def kvq():
    from fp8_quantized_paged_concat_gb300 import _build
    _build.build()
    import fp8_quantized_paged_concat_gb300 as m
    m.load_library()
    return m


def test_noalloc_split_decode_matches_the_workspace_entry_point(kvq, oracle_mod):
    from test_gpu_attention import check, host_cache

    for call, (tokens, topk, splits, seed) in enumerate(((4, 1024, 8, 551), (6, 700, 5, 552))):
        w = wl.make_attention(f"no-alloc call {call}", tokens, 128, topk, 32, 64, seed, p_unused=0.1)
        cache = host_cache(oracle_mod, w.fill)
        dcache = torch.from_numpy(cache).to(DEV)
        q, idx = w.q.to(DEV), w.indices.to(DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        out, lse = kvq.kvq_sparse_mla_attention_split_nvfp4_ds_mla_noalloc(q, idx, dcache, w.softmax_scale,
                                                                           num_splits=splits, status=status)
        ref_out, ref_lse = kvq.kvq_sparse_mla_attention_split_nvfp4_ds_mla(q, idx, dcache, w.softmax_scale,
                                                                           num_splits=splits)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), f"call {call}: out differs"
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32)), f"call {call}: lse differs"
        check(oracle_mod, cache, w.q, wl.host(w.indices), w.softmax_scale, out, lse)


def test_noalloc_refuses_more_rows_than_the_array_holds(kvq):
    rows = kvq.NOALLOC_SCRATCH_BYTES // (514 * 4)
    tokens = rows // (128 * 32) + 1                   # 128 heads x 32 ranges: one token too many
    q = torch.zeros((tokens, 128, 576), dtype=torch.bfloat16, device=DEV)
    idx = torch.full((tokens, 2048), -1, dtype=torch.int32, device=DEV)
    cache = torch.zeros((4, 64, 352), dtype=torch.uint8, device=DEV)
    with pytest.raises(RuntimeError, match="more than the library's fixed"):
        kvq.kvq_sparse_mla_attention_split_nvfp4_ds_mla_noalloc(q, idx, cache, 0.05, num_splits=32)
