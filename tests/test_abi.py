"""The C ABI library on a host without a GPU: it builds, loads, exports every
entry point include/kvq.h declares, and rejects bad arguments on the host
before any CUDA call.  No kernel is launched here.

The argument-rejection tests pass fake device addresses; they are skipped
where a GPU is visible, so that a validation gap could never turn into a
launch on a real device.
"""
import os
import re
import subprocess

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")

no_gpu_only = pytest.mark.skipif(torch.cuda.is_available(),
                                 reason="fake-pointer validation tests run only on GPU-less hosts")


@pytest.fixture(scope="module")
def lib():
    from fp8_quantized_paged_concat_gb300 import _build
    import fp8_quantized_paged_concat_gb300 as kvq
    _build.build()
    return kvq.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_hot_path_calls():
    names = declared_functions()
    for n in ("kvq_write_nvfp4_ds_mla", "kvq_gather_upconvert_nvfp4_ds_mla",
              "kvq_gather_upconvert_fp8_ds_mla", "kvq_reshape_and_cache_nvfp4"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from fp8_quantized_paged_concat_gb300 import library_path
    out = subprocess.run(["nm", "-D", "--defined-only", library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (kvq_[a-z0-9_]+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)
    assert lib.kvq_version() == 100


def test_library_is_built_for_sm_103a_only():
    from fp8_quantized_paged_concat_gb300 import _build
    assert "arch=compute_103a,code=sm_103a" in _build.ARCH
    assert not any("fast-math" in f or "fast_math" in f for f in _build.NVCC_FLAGS)


A = 0x10000000          # a 256-byte-aligned fake device address, never dereferenced


def err(lib):
    return lib.kvq_last_error_string().decode()


def write_args(entry=352, **over):
    args = dict(kv_c=A, kv_c_stride=512, k_pe=A, k_pe_stride=64, slot_mapping=A, num_tokens=16,
                kv_cache=A, num_blocks=4, block_size=64, block_stride=64 * entry,
                entry_stride=entry, d_status=None, stream=None)
    args.update(over)
    return list(args.values())


@no_gpu_only
@pytest.mark.parametrize("fn,entry", [("kvq_write_nvfp4_ds_mla", 352), ("kvq_write_fp8_ds_mla", 656)])
@pytest.mark.parametrize("over,needle", [
    (dict(num_tokens=-1), "num_tokens < 0"),
    (dict(kv_c=None), "kv_c is NULL"),
    (dict(kv_c=A + 8), "kv_c must be 16-byte aligned"),
    (dict(kv_c_stride=500), "row stride"),
    (dict(kv_c_stride=516), "row stride"),
    (dict(k_pe_stride=60), "row stride"),
    (dict(slot_mapping=None), "slot_mapping is NULL"),
    (dict(kv_cache=A + 4), "16-byte aligned"),
    (dict(entry_stride=336), "entry_stride"),
    (dict(entry_stride=664), "entry_stride"),
    (dict(block_stride=100), "block_stride"),
    (dict(num_blocks=0), "positive"),
    (dict(block_size=0), "positive"),
])
def test_write_rejects_bad_arguments_on_host(lib, fn, entry, over, needle):
    assert getattr(lib, fn)(*write_args(entry, **over)) == 1
    assert needle in err(lib), err(lib)


def gather_args(**over):
    args = dict(src_cache=A, num_blocks=4, block_size=64, block_stride=64 * 352, entry_stride=352,
                dst=A, dst_stride=576, num_out_tokens=100, block_table=A, block_table_stride=3,
                block_table_width=3, workspace_starts=A, seq_starts=A, batch_size=2,
                d_status=None, stream=None)
    args.update(over)
    return list(args.values())


@no_gpu_only
@pytest.mark.parametrize("over,needle", [
    (dict(num_out_tokens=-5), "num_out_tokens < 0"),
    (dict(num_out_tokens=1 << 31), "int32"),
    (dict(src_cache=None), "cache is NULL"),
    (dict(dst=A + 2), "dst must be 16-byte aligned"),
    (dict(dst_stride=575), "row stride"),
    (dict(batch_size=0), "batch_size"),
    (dict(block_table=None), "non-NULL"),
    (dict(seq_starts=None), "non-NULL"),
    (dict(workspace_starts=A + 2), "4-byte aligned"),
    (dict(block_table_width=0), "block_table_width"),
    (dict(block_table_stride=2), "block_table_stride"),
    (dict(entry_stride=336), "entry_stride"),
])
def test_gather_rejects_bad_arguments_on_host(lib, over, needle):
    assert lib.kvq_gather_upconvert_nvfp4_ds_mla(*gather_args(**over)) == 1
    assert needle in err(lib), err(lib)


@no_gpu_only
def test_fp8_gather_requires_656_byte_entries(lib):
    args = gather_args(entry_stride=352)
    assert lib.kvq_gather_upconvert_fp8_ds_mla(*args) == 1
    assert "656" in err(lib)


def per_head_args(**over):
    args = dict(key=A, value=A, kst=1024, ksh=128, vst=1024, vsh=128, slot_mapping=A,
                num_tokens=8, num_heads=8, head_size=128, kv_cache=A, num_pages=4, block_size=16,
                layout=0, k_scale=A, v_scale=A, d_status=None, stream=None)
    args.update(over)
    return list(args.values())


@no_gpu_only
@pytest.mark.parametrize("over,needle", [
    (dict(num_tokens=-1), "num_tokens < 0"),
    (dict(head_size=72), "multiple of 16"),
    (dict(num_heads=0), "num_heads"),
    (dict(key=None), "NULL"),
    (dict(value=A + 8), "16-byte aligned"),
    (dict(ksh=100), "multiples of 8"),
    (dict(k_scale=None), "fp32 scalars"),
    (dict(kv_cache=A + 8), "16-byte aligned"),
    (dict(num_pages=0), "positive"),
    (dict(head_size=16, num_heads=1, block_size=1), "multiple of 8"),
    (dict(layout=2), "KVQ_LAYOUT_NHD (0) or KVQ_LAYOUT_HND (1)"),
    (dict(layout=-1), "layout must be"),
])
def test_per_head_rejects_bad_arguments_on_host(lib, over, needle):
    assert lib.kvq_reshape_and_cache_nvfp4(*per_head_args(**over)) == 1
    assert needle in err(lib), err(lib)


@no_gpu_only
def test_zero_sized_calls_are_noops_without_device(lib):
    assert lib.kvq_write_nvfp4_ds_mla(*write_args(num_tokens=0, kv_c=None)) == 0
    assert lib.kvq_gather_upconvert_fp8_ds_mla(*gather_args(num_out_tokens=0, dst=None)) == 0
    assert lib.kvq_reshape_and_cache_nvfp4(*per_head_args(num_tokens=0)) == 0
    assert lib.kvq_selftest_convert(0, 0, None, None, None, None, None, None) == 0


@no_gpu_only
def test_valid_arguments_without_a_gpu_report_a_cuda_error(lib):
    """With no device the call fails cleanly at the device query."""
    assert lib.kvq_write_nvfp4_ds_mla(*write_args()) == 3
    assert "kvq_write_nvfp4_ds_mla" in err(lib)


def index_args(**over):
    args = dict(req_id=A, num_req_ids=10, token_indices=A, num_tokens=10, topk=8, ti_stride=8,
                block_table=A, bt_stride=4, bt_width=4, num_requests=2, block_size=16,
                num_blocks=64, out=A, out_stride=8, d_status=None, stream=None)
    args.update(over)
    return list(args.values())


@no_gpu_only
@pytest.mark.parametrize("over,needle", [
    (dict(num_req_ids=11), "req_id has 11 entries but token_indices has 10 rows"),
    (dict(num_req_ids=9), "req_id has 9 entries"),
    (dict(topk=-1), "< 0"),
    (dict(out=None), "non-NULL"),
    (dict(ti_stride=4), "row strides"),
    (dict(num_requests=0), "num_requests"),
    (dict(num_blocks=1 << 30, block_size=16), "int32 slot"),
])
def test_index_conversion_rejects_bad_arguments_on_host(lib, over, needle):
    assert lib.kvq_req_index_to_global_slot(*index_args(**over)) == 1
    assert needle in err(lib), err(lib)


@no_gpu_only
def test_index_conversion_zero_sized_is_noop(lib):
    assert lib.kvq_req_index_to_global_slot(*index_args(num_tokens=0, num_req_ids=0, req_id=None)) == 0


def dequant_args(**over):
    args = dict(kv_cache=A, num_pages=4, block_size=16, layout=1, num_heads=8, head_size=128, slot_mapping=A,
                num_tokens=8, k_scale=A, v_scale=A, key_out=A, kst=1024, ksh=128, value_out=A,
                vst=1024, vsh=128, d_status=None, stream=None)
    args.update(over)
    return list(args.values())


@no_gpu_only
@pytest.mark.parametrize("over,needle", [
    (dict(head_size=40), "multiple of 16"),
    (dict(key_out=None), "NULL"),
    (dict(ksh=64), "overlap"),
    (dict(vst=512), "overlap"),
    (dict(kv_cache=A + 4), "16-byte aligned"),
    (dict(layout=7), "layout must be"),
])
def test_dequant_rejects_bad_arguments_on_host(lib, over, needle):
    assert lib.kvq_dequant_nvfp4_per_head(*dequant_args(**over)) == 1
    assert needle in err(lib), err(lib)


def attention_args(**over):
    args = dict(q=A, qst=128 * 576, qsh=576, num_tokens=4, num_heads=128, indices=A, istride=64,
                topk=64, kv_cache=A, num_blocks=8, block_size=64, block_stride=64 * 352,
                entry_stride=352, scale=0.05, out=A, ost=128 * 512, osh=512, lse=A, lst=128,
                d_status=None, stream=None)
    args.update(over)
    return list(args.values())


@no_gpu_only
@pytest.mark.parametrize("over,needle", [
    (dict(num_heads=0), "num_heads must be in [1, 128]"),
    (dict(num_heads=129), "num_heads must be in [1, 128]"),
    (dict(q=None), "non-NULL"),
    (dict(out=A + 8), "16-byte aligned"),
    (dict(qsh=512), "head stride >= 576"),
    (dict(osh=512, ost=500), "must not overlap"),
    (dict(lst=100), "lse"),
    (dict(istride=32), "stride >= topk"),
    (dict(scale=float("inf")), "finite"),
    (dict(scale=float("nan")), "finite"),
    (dict(entry_stride=336), "entry_stride"),
    (dict(topk=-1), "< 0"),
])
def test_attention_rejects_bad_arguments_on_host(lib, over, needle):
    assert lib.kvq_sparse_mla_attention_nvfp4_ds_mla(*attention_args(**over)) == 1
    assert needle in err(lib), err(lib)


@no_gpu_only
def test_attention_zero_tokens_is_noop(lib):
    assert lib.kvq_sparse_mla_attention_nvfp4_ds_mla(*attention_args(num_tokens=0, q=None)) == 0


@no_gpu_only
def test_fp8_attention_requires_656_byte_entries(lib):
    assert lib.kvq_sparse_mla_attention_fp8_ds_mla(*attention_args(entry_stride=352, block_stride=64 * 352)) == 1
    assert "656" in err(lib), err(lib)


def split_args(num_splits=4, workspace=A, workspace_bytes=1 << 30, **over):
    args = attention_args(**over)
    return args[:-2] + [num_splits, workspace, workspace_bytes] + args[-2:]


@no_gpu_only
@pytest.mark.parametrize("over,needle", [
    (dict(num_splits=0), "num_splits must be in [1, 32]"),
    (dict(num_splits=33), "num_splits must be in [1, 32]"),
    (dict(workspace=None), "workspace"),
    (dict(workspace=A + 8), "workspace"),
    (dict(workspace_bytes=4 * 128 * 4 * 514 * 4 - 16), "at least 4210688 bytes"),
    (dict(num_heads=129), "num_heads must be in [1, 128]"),
])
def test_split_attention_rejects_bad_arguments_on_host(lib, over, needle):
    assert lib.kvq_sparse_mla_attention_split_nvfp4_ds_mla(*split_args(**over)) == 1
    assert needle in err(lib), err(lib)


def test_split_workspace_bytes(lib):
    f = lib.kvq_sparse_mla_attention_split_workspace_bytes
    assert f(4, 128, 4) == 4 * 128 * 4 * 514 * 4
    assert f(1, 1, 1) == 2064                          # 2056 rounded up to 16
    assert f(0, 128, 8) == 0
    assert f(-1, 128, 8) == -1 and f(4, 0, 8) == -1 and f(4, 128, 0) == -1
    assert f(1 << 62, 128, 32) == -1                  # past INT64_MAX


@no_gpu_only
def test_split_attention_one_range_needs_no_workspace(lib):
    """One range is the plain entry point: no workspace needed; without a
    device the call passes the argument checks and fails at the device query."""
    assert lib.kvq_sparse_mla_attention_split_nvfp4_ds_mla(*split_args(num_splits=1, workspace=None,
                                                                        workspace_bytes=0)) == 3
    assert "kvq_sparse_mla_attention_split_nvfp4_ds_mla" in err(lib)


@no_gpu_only
def test_noalloc_split_refuses_oversized_calls_on_host(lib):
    """128 heads x 32 ranges x 3 tokens need more than the fixed array holds."""
    args = attention_args(num_tokens=3, ost=128 * 512)
    args = args[:-2] + [32] + args[-2:]
    assert lib.kvq_sparse_mla_attention_split_nvfp4_ds_mla_noalloc(*args) == 1
    assert "more than the library's fixed 25165824-byte array" in err(lib), err(lib)


def prefill_split_args(**over):
    args = dict(q=A, qst=16 * 576, qsh=576, num_tokens=8, num_heads=16, query_start=A, context_lens=A,
                batch_size=2, max_query_len=4, block_table=A, bt_stride=8, bt_width=8, kv_cache=A,
                num_blocks=16, block_size=64, block_stride=64 * 352, entry_stride=352, scale=0.05, out=A,
                ost=16 * 512, osh=512, lse=A, lst=16, max_context_len=500, num_splits=4, workspace=A,
                workspace_bytes=1 << 30, d_status=None, stream=None)
    args.update(over)
    return list(args.values())


@no_gpu_only
@pytest.mark.parametrize("over,needle", [
    (dict(num_splits=0), "num_splits must be in [1, 32]"),
    (dict(num_splits=33), "num_splits must be in [1, 32]"),
    (dict(workspace=None), "workspace"),
    (dict(workspace_bytes=8 * 16 * 4 * 514 * 4 - 16), "at least 1052672 bytes"),
    (dict(max_context_len=-1), "max_context_len"),
])
def test_prefill_split_rejects_bad_arguments_on_host(lib, over, needle):
    assert lib.kvq_prefill_mla_attention_split_nvfp4_ds_mla(*prefill_split_args(**over)) == 1
    assert needle in err(lib), err(lib)


@no_gpu_only
def test_prefill_split_valid_arguments_reach_the_device_check(lib):
    assert lib.kvq_prefill_mla_attention_split_fp8_ds_mla(*prefill_split_args(entry_stride=656,
                                                                              block_stride=64 * 656)) == 3
