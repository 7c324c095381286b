"""GB300 quantized paged KV-cache write and gather-upconvert.

Thin Python binding over libkvq.so (include/kvq.h): each function has the
name of the C entry point, checks dtypes / devices / shapes of the torch
tensors it is given, passes their data pointers and strides and the current
CUDA stream, and raises RuntimeError on a non-OK status.  Every step of the
computation runs in the library's sm_103a kernels; there is no fallback.  The
library is built by ``__graft_entry__.build()`` (or
``python -m fp8_quantized_paged_concat_gb300._build``); importing this
package does not load it, the first call does, and fails loudly if it is
missing.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "kvq_write_nvfp4_ds_mla", "kvq_write_fp8_ds_mla", "kvq_gather_upconvert_nvfp4_ds_mla",
    "kvq_gather_upconvert_fp8_ds_mla", "kvq_reshape_and_cache_nvfp4", "kvq_selftest_convert",
    "kvq_dequant_nvfp4_per_head", "kvq_req_index_to_global_slot",
    "kvq_sparse_mla_attention_nvfp4_ds_mla", "kvq_sparse_mla_attention_fp8_ds_mla",
    "kvq_prefill_mla_attention_nvfp4_ds_mla", "kvq_prefill_mla_attention_fp8_ds_mla",
    "kvq_sparse_mla_attention_split_nvfp4_ds_mla", "kvq_sparse_mla_attention_split_fp8_ds_mla",
    "kvq_sparse_mla_attention_split_workspace_bytes", "default_num_splits", "ATTN_MAX_SPLITS",
    "kvq_sparse_mla_attention_split_nvfp4_ds_mla_noalloc", "NOALLOC_SCRATCH_BYTES",
    "kvq_prefill_mla_attention_split_nvfp4_ds_mla", "kvq_prefill_mla_attention_split_fp8_ds_mla",
    "default_prefill_num_splits", "kvq_prefill_mla_attention_workspace",
    "kvq_last_error_string", "kvq_version", "library_path", "load_library",
    "NVFP4_DS_MLA_ENTRY_BYTES", "FP8_DS_MLA_ENTRY_BYTES", "STATUS_BAD_INDEX", "STATUS_BAD_BATCH",
    "STATUS_TIMEOUT",
    "nvfp4_full_dim",
]

NVFP4_DS_MLA_ENTRY_BYTES = 352
FP8_DS_MLA_ENTRY_BYTES = 656
STATUS_BAD_INDEX = 0x1
STATUS_BAD_BATCH = 0x2
STATUS_TIMEOUT = 0x4
ATTN_MAX_SPLITS = 32
NOALLOC_SCRATCH_BYTES = 24 << 20

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_U32 = ctypes.c_uint32

_SIGNATURES = {
    "kvq_write_nvfp4_ds_mla": [_P, _I64, _P, _I64, _P, _I64, _P, _I64, _I32, _I64, _I64, _P, _P],
    "kvq_write_fp8_ds_mla": [_P, _I64, _P, _I64, _P, _I64, _P, _I64, _I32, _I64, _I64, _P, _P],
    "kvq_gather_upconvert_nvfp4_ds_mla": [_P, _I64, _I32, _I64, _I64, _P, _I64, _I64, _P, _I64,
                                          _I32, _P, _P, _I32, _P, _P],
    "kvq_gather_upconvert_fp8_ds_mla": [_P, _I64, _I32, _I64, _I64, _P, _I64, _I64, _P, _I64,
                                        _I32, _P, _P, _I32, _P, _P],
    "kvq_reshape_and_cache_nvfp4": [_P, _P, _I64, _I64, _I64, _I64, _P, _I64, _I32, _I32, _P, _I64,
                                    _I32, _I32, _P, _P, _P, _P],
    "kvq_selftest_convert": [_U32, _I64, _P, _P, _P, _P, _P, _P],
    "kvq_dequant_nvfp4_per_head": [_P, _I64, _I32, _I32, _I32, _I32, _P, _I64, _P, _P, _P, _I64, _I64, _P,
                                   _I64, _I64, _P, _P],
    "kvq_req_index_to_global_slot": [_P, _I64, _P, _I64, _I32, _I64, _P, _I64, _I32, _I32, _I32, _I64,
                                     _P, _I64, _P, _P],
    "kvq_sparse_mla_attention_nvfp4_ds_mla": [_P, _I64, _I64, _I64, _I32, _P, _I64, _I32, _P, _I64, _I32,
                                              _I64, _I64, ctypes.c_float, _P, _I64, _I64, _P, _I64,
                                              _P, _P],
    "kvq_sparse_mla_attention_fp8_ds_mla": [_P, _I64, _I64, _I64, _I32, _P, _I64, _I32, _P, _I64, _I32,
                                            _I64, _I64, ctypes.c_float, _P, _I64, _I64, _P, _I64,
                                            _P, _P],
    "kvq_prefill_mla_attention_nvfp4_ds_mla": [_P, _I64, _I64, _I64, _I32, _P, _P, _I32, _I32, _P, _I64, _I32,
                                               _P, _I64, _I32, _I64, _I64, ctypes.c_float, _P, _I64, _I64, _P,
                                               _I64, _P, _P],
    "kvq_prefill_mla_attention_fp8_ds_mla": [_P, _I64, _I64, _I64, _I32, _P, _P, _I32, _I32, _P, _I64, _I32,
                                             _P, _I64, _I32, _I64, _I64, ctypes.c_float, _P, _I64, _I64, _P,
                                             _I64, _P, _P],
    "kvq_sparse_mla_attention_split_nvfp4_ds_mla": [_P, _I64, _I64, _I64, _I32, _P, _I64, _I32, _P, _I64, _I32,
                                                    _I64, _I64, ctypes.c_float, _P, _I64, _I64, _P, _I64,
                                                    _I32, _P, _I64, _P, _P],
    "kvq_sparse_mla_attention_split_fp8_ds_mla": [_P, _I64, _I64, _I64, _I32, _P, _I64, _I32, _P, _I64, _I32,
                                                  _I64, _I64, ctypes.c_float, _P, _I64, _I64, _P, _I64,
                                                  _I32, _P, _I64, _P, _P],
    "kvq_prefill_mla_attention_split_nvfp4_ds_mla": [_P, _I64, _I64, _I64, _I32, _P, _P, _I32, _I32, _P, _I64,
                                                     _I32, _P, _I64, _I32, _I64, _I64, ctypes.c_float, _P, _I64,
                                                     _I64, _P, _I64, _I32, _I32, _P, _I64, _P, _P],
    "kvq_prefill_mla_attention_split_fp8_ds_mla": [_P, _I64, _I64, _I64, _I32, _P, _P, _I32, _I32, _P, _I64,
                                                   _I32, _P, _I64, _I32, _I64, _I64, ctypes.c_float, _P, _I64,
                                                   _I64, _P, _I64, _I32, _I32, _P, _I64, _P, _P],
    "kvq_prefill_mla_attention_workspace": [_P, _I64, _I64, _I64, _I32, _P, _P, _P, _I32, _I32, _P, _I64, _I64,
                                            ctypes.c_float, _P, _I64, _I64, _P, _I64, _P, _P],
    "kvq_sparse_mla_attention_split_nvfp4_ds_mla_noalloc": [_P, _I64, _I64, _I64, _I32, _P, _I64, _I32, _P, _I64,
                                                            _I32, _I64, _I64, ctypes.c_float, _P, _I64, _I64, _P,
                                                            _I64, _I32, _P, _P],
}


def library_path() -> str:
    return os.path.join(_HERE, "_lib", "libkvq.so")


def load_library():
    """Loads libkvq.so (once).  Raises RuntimeError if it has not been built."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                               "(there is no CPU fallback)")
        handle = ctypes.CDLL(path)
        for name, argtypes in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.argtypes = argtypes
            fn.restype = _I32
        handle.kvq_last_error_string.restype = ctypes.c_char_p
        handle.kvq_last_error_string.argtypes = []
        handle.kvq_version.restype = _I32
        handle.kvq_version.argtypes = []
        handle.kvq_sparse_mla_attention_split_workspace_bytes.restype = _I64
        handle.kvq_sparse_mla_attention_split_workspace_bytes.argtypes = [_I64, _I32, _I32]
        _lib = handle
    return _lib


def kvq_last_error_string() -> str:
    return load_library().kvq_last_error_string().decode()


def kvq_version() -> int:
    return load_library().kvq_version()


def nvfp4_full_dim(head_size: int) -> int:
    """Last dimension of the per-head NVFP4 cache: head_size/2 + head_size/16."""
    return head_size // 2 + head_size // 16


def _call(name: str, *args):
    status = getattr(load_library(), name)(*args)
    if status != 0:
        raise RuntimeError(f"{name} failed (status {status}): {kvq_last_error_string()}")


def _stream(stream, device) -> int:
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


def _status_ptr(status):
    if status is None:
        return None
    if status.dtype != torch.int32 or not status.is_cuda or status.numel() < 1:
        raise ValueError("status must be a CUDA int32 tensor with at least one element")
    return status.data_ptr()


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _bf16_rows(name, t, width):
    _need(t.dtype == torch.bfloat16 and t.is_cuda and t.dim() == 2 and t.shape[1] >= width
          and t.stride(1) == 1, f"{name}: expected a CUDA bf16 [T, >={width}] tensor with unit inner stride")


def _mla_cache(name, t, entry):
    _need(t.dtype == torch.uint8 and t.is_cuda and t.dim() == 3 and t.shape[2] >= entry
          and t.stride(2) == 1, f"{name}: expected a CUDA uint8 [num_blocks, block_size, >={entry}] tensor")


def _write(cname, entry, kv_c, k_pe, kv_cache, slot_mapping, status, stream):
    _bf16_rows("kv_c", kv_c, 512)
    _bf16_rows("k_pe", k_pe, 64)
    _mla_cache("kv_cache", kv_cache, entry)
    _need(slot_mapping.dtype == torch.int64 and slot_mapping.is_cuda and slot_mapping.dim() == 1
          and slot_mapping.is_contiguous(), "slot_mapping: expected a contiguous CUDA int64 vector")
    T = slot_mapping.shape[0]
    _need(kv_c.shape[0] >= T and k_pe.shape[0] >= T, "kv_c / k_pe have fewer rows than slot_mapping")
    _call(cname, kv_c.data_ptr(), kv_c.stride(0), k_pe.data_ptr(), k_pe.stride(0),
          slot_mapping.data_ptr(), T, kv_cache.data_ptr(), kv_cache.shape[0], kv_cache.shape[1],
          kv_cache.stride(0), kv_cache.stride(1), _status_ptr(status), _stream(stream, kv_cache.device))


def kvq_write_nvfp4_ds_mla(kv_c, k_pe, kv_cache, slot_mapping, status=None, stream=None):
    """Writes 352-byte nvfp4_ds_mla entries: kv_c bf16 [T, 512], k_pe bf16
    [T, 64], kv_cache uint8 [num_blocks, block_size, >=352], slot_mapping
    int64 [T] (negative = padding).  Asynchronous on ``stream``."""
    _write("kvq_write_nvfp4_ds_mla", 352, kv_c, k_pe, kv_cache, slot_mapping, status, stream)


def kvq_write_fp8_ds_mla(kv_c, k_pe, kv_cache, slot_mapping, status=None, stream=None):
    """Writes 656-byte fp8_ds_mla entries (arguments as kvq_write_nvfp4_ds_mla)."""
    _write("kvq_write_fp8_ds_mla", 656, kv_c, k_pe, kv_cache, slot_mapping, status, stream)


def _gather(cname, entry, src_cache, dst, block_table, workspace_starts, seq_starts, batch_size,
            status, stream):
    _mla_cache("src_cache", src_cache, entry)
    _bf16_rows("dst", dst, 576)
    for name, t in (("block_table", block_table), ("workspace_starts", workspace_starts),
                    ("seq_starts", seq_starts)):
        _need(t.dtype == torch.int32 and t.is_cuda, f"{name}: expected a CUDA int32 tensor")
    _need(block_table.dim() == 2 and block_table.stride(1) == 1, "block_table: expected [B, W] rows")
    _need(workspace_starts.is_contiguous() and seq_starts.is_contiguous(),
          "workspace_starts / seq_starts must be contiguous")
    B = int(seq_starts.shape[0]) if batch_size is None else int(batch_size)
    _need(B <= seq_starts.shape[0] and B <= workspace_starts.shape[0] and B <= block_table.shape[0],
          "batch_size exceeds the metadata tensors")
    _call(cname, src_cache.data_ptr(), src_cache.shape[0], src_cache.shape[1], src_cache.stride(0),
          src_cache.stride(1), dst.data_ptr(), dst.stride(0), dst.shape[0], block_table.data_ptr(),
          block_table.stride(0), block_table.shape[1], workspace_starts.data_ptr(),
          seq_starts.data_ptr(), B, _status_ptr(status), _stream(stream, dst.device))


def kvq_gather_upconvert_nvfp4_ds_mla(src_cache, dst, block_table, workspace_starts, seq_starts,
                                      batch_size=None, status=None, stream=None):
    """Gathers nvfp4_ds_mla pages into dst bf16 [T, 576] (T = dst rows):
    block_table int32 [B, W], workspace_starts / seq_starts int32 [B]."""
    _gather("kvq_gather_upconvert_nvfp4_ds_mla", 352, src_cache, dst, block_table,
            workspace_starts, seq_starts, batch_size, status, stream)


def kvq_gather_upconvert_fp8_ds_mla(src_cache, dst, block_table, workspace_starts, seq_starts,
                                    batch_size=None, status=None, stream=None):
    """Gathers fp8_ds_mla pages into dst bf16 [T, 576] (as the nvfp4 gather)."""
    _gather("kvq_gather_upconvert_fp8_ds_mla", 656, src_cache, dst, block_table,
            workspace_starts, seq_starts, batch_size, status, stream)


def kvq_reshape_and_cache_nvfp4(key, value, kv_cache, slot_mapping, k_scale, v_scale,
                                status=None, stream=None, layout="NHD"):
    """Writes the per-head NVFP4 cache uint8 [P, 2, block_size, H, full_dim]
    (layout "NHD") or [P, 2, H, block_size, full_dim] ("HND") from key / value
    bf16 [T, H, D]; k_scale / v_scale CUDA fp32 scalars."""
    for name, t in (("key", key), ("value", value)):
        _need(t.dtype == torch.bfloat16 and t.is_cuda and t.dim() == 3 and t.stride(2) == 1,
              f"{name}: expected a CUDA bf16 [T, H, D] tensor with unit inner stride")
    _need(key.shape == value.shape, "key and value shapes differ")
    T, H, D = key.shape
    code, block_size = _per_head_cache(kv_cache, H, D, layout)
    _need(slot_mapping.dtype == torch.int64 and slot_mapping.is_cuda and slot_mapping.is_contiguous()
          and slot_mapping.shape[0] == T, "slot_mapping: expected a contiguous CUDA int64 [T]")
    for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        _need(t.dtype == torch.float32 and t.is_cuda and t.numel() >= 1, f"{name}: CUDA fp32 scalar")
    _call("kvq_reshape_and_cache_nvfp4", key.data_ptr(), value.data_ptr(), key.stride(0),
          key.stride(1), value.stride(0), value.stride(1), slot_mapping.data_ptr(), T, H, D,
          kv_cache.data_ptr(), kv_cache.shape[0], block_size, code, k_scale.data_ptr(),
          v_scale.data_ptr(), _status_ptr(status), _stream(stream, kv_cache.device))


LAYOUTS = {"NHD": 0, "HND": 1}


def _per_head_cache(kv_cache, H, D, layout):
    """Checks the per-head cache tensor; returns (layout code, block_size)."""
    _need(layout in LAYOUTS, f"layout: expected one of {sorted(LAYOUTS)}, got {layout!r}")
    code = LAYOUTS[layout]
    head_axis = 3 if code == 0 else 2
    shape = "[P, 2, block_size, H, D/2 + D/16]" if code == 0 else "[P, 2, H, block_size, D/2 + D/16]"
    _need(kv_cache.dtype == torch.uint8 and kv_cache.is_cuda and kv_cache.dim() == 5
          and kv_cache.is_contiguous() and kv_cache.shape[1] == 2 and kv_cache.shape[head_axis] == H
          and kv_cache.shape[4] == nvfp4_full_dim(D),
          f"kv_cache: expected a contiguous CUDA uint8 {shape} tensor for layout {layout}")
    return code, kv_cache.shape[5 - head_axis]


def kvq_dequant_nvfp4_per_head(kv_cache, slot_mapping, k_scale, v_scale, key_out, value_out,
                               status=None, stream=None, layout="NHD"):
    """Reads the per-head NVFP4 cache (layout "NHD" or "HND") back at
    slot_mapping into key_out / value_out bf16 [T, H, D] (rows of padding
    slots are left untouched)."""
    for name, t in (("key_out", key_out), ("value_out", value_out)):
        _need(t.dtype == torch.bfloat16 and t.is_cuda and t.dim() == 3 and t.stride(2) == 1,
              f"{name}: expected a CUDA bf16 [T, H, D] tensor with unit inner stride")
    _need(key_out.shape == value_out.shape, "key_out and value_out shapes differ")
    T, H, D = key_out.shape
    code, block_size = _per_head_cache(kv_cache, H, D, layout)
    _need(slot_mapping.dtype == torch.int64 and slot_mapping.is_cuda and slot_mapping.is_contiguous()
          and slot_mapping.shape[0] == T, "slot_mapping: expected a contiguous CUDA int64 [T]")
    for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        _need(t.dtype == torch.float32 and t.is_cuda and t.numel() >= 1, f"{name}: CUDA fp32 scalar")
    _call("kvq_dequant_nvfp4_per_head", kv_cache.data_ptr(), kv_cache.shape[0], block_size, code, H, D,
          slot_mapping.data_ptr(), T, k_scale.data_ptr(), v_scale.data_ptr(), key_out.data_ptr(),
          key_out.stride(0), key_out.stride(1), value_out.data_ptr(), value_out.stride(0),
          value_out.stride(1), _status_ptr(status), _stream(stream, kv_cache.device))


def kvq_req_index_to_global_slot(req_id, token_indices, block_table, block_size: int, num_blocks: int,
                                 out=None, status=None, stream=None):
    """Sparse-decode index conversion: int32 token_indices [N, topk] of
    requests req_id [N] -> global slots int32 [N, topk] (-1 where unused).
    Raises RuntimeError when req_id and token_indices lengths differ."""
    for name, t in (("req_id", req_id), ("token_indices", token_indices), ("block_table", block_table)):
        _need(t.dtype == torch.int32 and t.is_cuda, f"{name}: expected a CUDA int32 tensor")
    _need(req_id.dim() == 1 and req_id.is_contiguous(), "req_id: expected a contiguous vector")
    _need(token_indices.dim() == 2 and token_indices.stride(1) == 1, "token_indices: expected [N, topk] rows")
    _need(block_table.dim() == 2 and block_table.stride(1) == 1, "block_table: expected [R, W] rows")
    N, topk = token_indices.shape
    if out is None:
        out = torch.empty((N, topk), dtype=torch.int32, device=token_indices.device)
    _need(out.dtype == torch.int32 and out.is_cuda and out.dim() == 2 and out.stride(1) == 1
          and tuple(out.shape) == (N, topk), "out: expected a CUDA int32 [N, topk] tensor")
    _call("kvq_req_index_to_global_slot", req_id.data_ptr(), req_id.shape[0], token_indices.data_ptr(),
          N, topk, token_indices.stride(0), block_table.data_ptr(), block_table.stride(0),
          block_table.shape[1], block_table.shape[0], block_size, num_blocks, out.data_ptr(),
          out.stride(0), _status_ptr(status), _stream(stream, token_indices.device))
    return out


def kvq_sparse_mla_attention_nvfp4_ds_mla(q, indices, kv_cache, softmax_scale: float, out=None, lse=None,
                                          status=None, stream=None):
    """Sparse MLA attention (MQA form) straight from the nvfp4_ds_mla cache:
    q bf16 [T, H, 576] (H <= 128), indices int32 [T, topk] global slots (< 0
    unused), kv_cache uint8 [num_blocks, block_size, >=352].  Returns (out
    bf16 [T, H, 512], lse fp32 [T, H]); lse=False skips the lse output."""
    return _attention("kvq_sparse_mla_attention_nvfp4_ds_mla", 352, q, indices, kv_cache, softmax_scale, out,
                      lse, status, stream)


def kvq_sparse_mla_attention_fp8_ds_mla(q, indices, kv_cache, softmax_scale: float, out=None, lse=None,
                                        status=None, stream=None):
    """The same attention straight from the 656-byte fp8_ds_mla cache."""
    return _attention("kvq_sparse_mla_attention_fp8_ds_mla", 656, q, indices, kv_cache, softmax_scale, out,
                      lse, status, stream)


def kvq_sparse_mla_attention_split_workspace_bytes(num_tokens: int, num_heads: int, num_splits: int) -> int:
    """Bytes of workspace the split-key decode needs (-1 for bad arguments)."""
    return load_library().kvq_sparse_mla_attention_split_workspace_bytes(num_tokens, num_heads, num_splits)


def default_num_splits(num_tokens: int, topk: int, device=None) -> int:
    """Key ranges per token for a decode batch of num_tokens: as many as one
    wave of CTAs holds (two CTAs per token and range, one CTA per SM), at
    most ATTN_MAX_SPLITS and at most one per 64-key tile, the count then
    trimmed so that no range is left empty."""
    if num_tokens <= 0:
        return 1
    sms = torch.cuda.get_device_properties(device if device is not None else torch.cuda.current_device()
                                           ).multi_processor_count
    tiles = (topk + 63) // 64
    want = max(1, min(ATTN_MAX_SPLITS, tiles, sms // (2 * num_tokens)))
    per_range = -(-tiles // want) if tiles else 1
    return max(1, -(-tiles // per_range)) if tiles else 1


def kvq_sparse_mla_attention_split_nvfp4_ds_mla(q, indices, kv_cache, softmax_scale: float, num_splits=None,
                                                workspace=None, out=None, lse=None, status=None, stream=None):
    """The sparse attention of kvq_sparse_mla_attention_nvfp4_ds_mla with each
    token's keys split into num_splits ranges (default: default_num_splits)
    whose partial results a second launch combines.  workspace: a CUDA uint8
    tensor of at least kvq_sparse_mla_attention_split_workspace_bytes bytes
    (allocated here when None)."""
    return _attention("kvq_sparse_mla_attention_split_nvfp4_ds_mla", 352, q, indices, kv_cache, softmax_scale, out,
                      lse, status, stream, split=(num_splits, workspace))


def kvq_sparse_mla_attention_split_fp8_ds_mla(q, indices, kv_cache, softmax_scale: float, num_splits=None,
                                              workspace=None, out=None, lse=None, status=None, stream=None):
    """The same split-key decode straight from the 656-byte fp8_ds_mla cache."""
    return _attention("kvq_sparse_mla_attention_split_fp8_ds_mla", 656, q, indices, kv_cache, softmax_scale, out,
                      lse, status, stream, split=(num_splits, workspace))


def kvq_sparse_mla_attention_split_nvfp4_ds_mla_noalloc(q, indices, kv_cache, softmax_scale: float, num_splits=None,
                                                        out=None, lse=None, status=None, stream=None):
    """The split-key decode with its partial results in the library's own
    fixed array (NOALLOC_SCRATCH_BYTES per GPU) instead of a workspace, for
    callers that cannot allocate device memory when they call in.  Calls that
    overlap on the GPU race on that array: order them."""
    return _attention("kvq_sparse_mla_attention_split_nvfp4_ds_mla_noalloc", 352, q, indices, kv_cache,
                      softmax_scale, out, lse, status, stream, split=(num_splits, "noalloc"))


def _attention(cname, entry, q, indices, kv_cache, softmax_scale, out, lse, status, stream, split=None):
    _need(q.dtype == torch.bfloat16 and q.is_cuda and q.dim() == 3 and q.shape[2] == 576
          and q.stride(2) == 1, "q: expected a CUDA bf16 [T, H, 576] tensor with unit inner stride")
    T, H = q.shape[0], q.shape[1]
    _need(indices.dtype == torch.int32 and indices.is_cuda and indices.dim() == 2
          and indices.shape[0] == T and (indices.shape[1] == 0 or indices.stride(1) == 1),
          "indices: expected CUDA int32 [T, topk] rows")
    _mla_cache("kv_cache", kv_cache, entry)
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q.device)
    _need(out.dtype == torch.bfloat16 and out.is_cuda and tuple(out.shape) == (T, H, 512)
          and out.stride(2) == 1, "out: expected a CUDA bf16 [T, H, 512] tensor with unit inner stride")
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    if lse is not False:
        _need(lse.dtype == torch.float32 and lse.is_cuda and tuple(lse.shape) == (T, H) and lse.stride(1) == 1,
              "lse: expected a CUDA fp32 [T, H] tensor with unit inner stride")
    args = [q.data_ptr(), q.stride(0), q.stride(1), T, H,
            indices.data_ptr(), max(indices.stride(0), indices.shape[1]), indices.shape[1], kv_cache.data_ptr(),
            kv_cache.shape[0], kv_cache.shape[1], kv_cache.stride(0), kv_cache.stride(1), float(softmax_scale),
            out.data_ptr(), out.stride(0), out.stride(1), None if lse is False else lse.data_ptr(),
            0 if lse is False else lse.stride(0)]
    if split is not None and split[1] == "noalloc":
        num_splits = split[0] if split[0] is not None else default_num_splits(T, indices.shape[1], q.device)
        args += [int(num_splits)]
    elif split is not None:
        num_splits, workspace = split
        if num_splits is None:
            num_splits = default_num_splits(T, indices.shape[1], q.device)
        need = kvq_sparse_mla_attention_split_workspace_bytes(T, H, num_splits) if num_splits > 1 else 0
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        if workspace is not None:
            _need(workspace.is_cuda and workspace.is_contiguous(), "workspace: expected a contiguous CUDA tensor")
        args += [int(num_splits), None if workspace is None else workspace.data_ptr(),
                 0 if workspace is None else workspace.numel() * workspace.element_size()]
    _call(cname, *args, _status_ptr(status), _stream(stream, q.device))
    return out, (None if lse is False else lse)


def kvq_prefill_mla_attention_nvfp4_ds_mla(q, query_start, context_lens, block_table, kv_cache,
                                           softmax_scale: float, max_query_len: int, out=None, lse=None,
                                           status=None, stream=None):
    """Dense prefill straight from the nvfp4_ds_mla cache: q bf16 [T, H, 576];
    request b's query tokens [query_start[b], query_start[b+1]) (int32 [B+1],
    at most max_query_len each) attend to its context positions [0,
    context_lens[b]) (int32 [B]) through block_table int32 [B, W].  Returns
    (out bf16 [T, H, 512], lse fp32 [T, H]); lse=False skips the lse output."""
    return _prefill("kvq_prefill_mla_attention_nvfp4_ds_mla", 352, q, query_start, context_lens, block_table,
                    kv_cache, softmax_scale, max_query_len, out, lse, status, stream)


def kvq_prefill_mla_attention_fp8_ds_mla(q, query_start, context_lens, block_table, kv_cache,
                                         softmax_scale: float, max_query_len: int, out=None, lse=None,
                                         status=None, stream=None):
    """The same dense prefill straight from the 656-byte fp8_ds_mla cache."""
    return _prefill("kvq_prefill_mla_attention_fp8_ds_mla", 656, q, query_start, context_lens, block_table,
                    kv_cache, softmax_scale, max_query_len, out, lse, status, stream)


def kvq_prefill_mla_attention_workspace(q, query_start, context_lens, workspace_starts, workspace,
                                        softmax_scale: float, max_query_len: int, out=None, lse=None, status=None,
                                        stream=None):
    """Dense prefill over a gathered bf16 workspace [R, >=576] (what
    kvq_gather_upconvert_*_ds_mla writes): request b's context position p is
    workspace row workspace_starts[b] + p, p < context_lens[b].  Returns
    (out bf16 [T, H, 512], lse fp32 [T, H]); lse=False skips the lse output."""
    _need(q.dtype == torch.bfloat16 and q.is_cuda and q.dim() == 3 and q.shape[2] == 576
          and q.stride(2) == 1, "q: expected a CUDA bf16 [T, H, 576] tensor with unit inner stride")
    T, H = q.shape[0], q.shape[1]
    B = context_lens.shape[0] if context_lens.dim() == 1 else -1
    for name, t, n in (("context_lens", context_lens, B), ("query_start", query_start, B + 1),
                       ("workspace_starts", workspace_starts, B)):
        _need(t.dtype == torch.int32 and t.is_cuda and t.dim() == 1 and t.shape[0] == n and t.is_contiguous(),
              f"{name}: expected a contiguous CUDA int32 vector of {n}")
    _need(workspace.dtype == torch.bfloat16 and workspace.is_cuda and workspace.dim() == 2
          and workspace.shape[1] >= 576 and workspace.stride(1) == 1,
          "workspace: expected a CUDA bf16 [R, >=576] tensor with unit inner stride")
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q.device)
    _need(out.dtype == torch.bfloat16 and out.is_cuda and tuple(out.shape) == (T, H, 512)
          and out.stride(2) == 1, "out: expected a CUDA bf16 [T, H, 512] tensor with unit inner stride")
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    if lse is not False:
        _need(lse.dtype == torch.float32 and lse.is_cuda and tuple(lse.shape) == (T, H) and lse.stride(1) == 1,
              "lse: expected a CUDA fp32 [T, H] tensor with unit inner stride")
    _call("kvq_prefill_mla_attention_workspace", q.data_ptr(), q.stride(0), q.stride(1), T, H,
          query_start.data_ptr(), context_lens.data_ptr(), workspace_starts.data_ptr(), B, int(max_query_len),
          workspace.data_ptr(), workspace.stride(0), workspace.shape[0], float(softmax_scale), out.data_ptr(),
          out.stride(0), out.stride(1), None if lse is False else lse.data_ptr(),
          0 if lse is False else lse.stride(0), _status_ptr(status), _stream(stream, q.device))
    return out, (None if lse is False else lse)


def default_prefill_num_splits(max_query_len: int, num_heads: int, batch_size: int, max_context_len: int,
                               device=None) -> int:
    """Context ranges per request for a dense prefill: as many as one wave
    of CTAs holds (two per 128-row block and range), at most
    ATTN_MAX_SPLITS and one per 64-position tile of the longest context."""
    blocks = -(-max_query_len * num_heads // 128) * batch_size
    if blocks <= 0:
        return 1
    sms = torch.cuda.get_device_properties(device if device is not None else torch.cuda.current_device()
                                           ).multi_processor_count
    tiles = (max_context_len + 63) // 64
    return max(1, min(ATTN_MAX_SPLITS, tiles, sms // (2 * blocks)))


def kvq_prefill_mla_attention_split_nvfp4_ds_mla(q, query_start, context_lens, block_table, kv_cache,
                                                 softmax_scale: float, max_query_len: int, max_context_len=None,
                                                 num_splits=None, workspace=None, out=None, lse=None, status=None,
                                                 stream=None):
    """The dense prefill of kvq_prefill_mla_attention_nvfp4_ds_mla with each
    request's context split into num_splits ranges sized from
    max_context_len (default: the longest context, read from the device)
    and combined by a second launch.  workspace as for the split decode
    (allocated here when None)."""
    return _prefill("kvq_prefill_mla_attention_split_nvfp4_ds_mla", 352, q, query_start, context_lens, block_table,
                    kv_cache, softmax_scale, max_query_len, out, lse, status, stream,
                    split=(max_context_len, num_splits, workspace))


def kvq_prefill_mla_attention_split_fp8_ds_mla(q, query_start, context_lens, block_table, kv_cache,
                                               softmax_scale: float, max_query_len: int, max_context_len=None,
                                               num_splits=None, workspace=None, out=None, lse=None, status=None,
                                               stream=None):
    """The same split dense prefill straight from the 656-byte fp8_ds_mla cache."""
    return _prefill("kvq_prefill_mla_attention_split_fp8_ds_mla", 656, q, query_start, context_lens, block_table,
                    kv_cache, softmax_scale, max_query_len, out, lse, status, stream,
                    split=(max_context_len, num_splits, workspace))


def _prefill(cname, entry, q, query_start, context_lens, block_table, kv_cache, softmax_scale, max_query_len,
             out, lse, status, stream, split=None):
    _need(q.dtype == torch.bfloat16 and q.is_cuda and q.dim() == 3 and q.shape[2] == 576
          and q.stride(2) == 1, "q: expected a CUDA bf16 [T, H, 576] tensor with unit inner stride")
    T, H = q.shape[0], q.shape[1]
    B = context_lens.shape[0] if context_lens.dim() == 1 else -1
    _need(context_lens.dtype == torch.int32 and context_lens.is_cuda and B >= 0 and context_lens.is_contiguous(),
          "context_lens: expected a contiguous CUDA int32 [B] tensor")
    _need(query_start.dtype == torch.int32 and query_start.is_cuda and tuple(query_start.shape) == (B + 1,)
          and query_start.is_contiguous(), "query_start: expected a contiguous CUDA int32 [B + 1] tensor")
    _need(block_table.dtype == torch.int32 and block_table.is_cuda and block_table.dim() == 2
          and block_table.shape[0] == B and block_table.stride(1) == 1,
          "block_table: expected a CUDA int32 [B, W] tensor with unit inner stride")
    _mla_cache("kv_cache", kv_cache, entry)
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q.device)
    _need(out.dtype == torch.bfloat16 and out.is_cuda and tuple(out.shape) == (T, H, 512)
          and out.stride(2) == 1, "out: expected a CUDA bf16 [T, H, 512] tensor with unit inner stride")
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    if lse is not False:
        _need(lse.dtype == torch.float32 and lse.is_cuda and tuple(lse.shape) == (T, H) and lse.stride(1) == 1,
              "lse: expected a CUDA fp32 [T, H] tensor with unit inner stride")
    args = [q.data_ptr(), q.stride(0), q.stride(1), T, H, query_start.data_ptr(), context_lens.data_ptr(),
            B, int(max_query_len), block_table.data_ptr(), block_table.stride(0), block_table.shape[1],
            kv_cache.data_ptr(), kv_cache.shape[0], kv_cache.shape[1], kv_cache.stride(0), kv_cache.stride(1),
            float(softmax_scale), out.data_ptr(), out.stride(0), out.stride(1),
            None if lse is False else lse.data_ptr(), 0 if lse is False else lse.stride(0)]
    if split is not None:
        max_context_len, num_splits, workspace = split
        if max_context_len is None:
            max_context_len = int(context_lens.max().item()) if B > 0 else 0
        if num_splits is None:
            num_splits = default_prefill_num_splits(int(max_query_len), H, B, max_context_len, q.device)
        need = kvq_sparse_mla_attention_split_workspace_bytes(T, H, num_splits) if num_splits > 1 else 0
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        if workspace is not None:
            _need(workspace.is_cuda and workspace.is_contiguous(), "workspace: expected a contiguous CUDA tensor")
        args += [int(max_context_len), int(num_splits), None if workspace is None else workspace.data_ptr(),
                 0 if workspace is None else workspace.numel() * workspace.element_size()]
    _call(cname, *args, _status_ptr(status), _stream(stream, q.device))
    return out, (None if lse is False else lse)


def kvq_selftest_convert(first_bits: int, count: int, device="cuda", stream=None):
    """Device converters over float32 bit patterns first_bits..+count-1:
    returns (e4m3_lo, e4m3_hi, e2m1_lo, e2m1_hi, bf16) CUDA tensors."""
    outs = [torch.empty(count, dtype=torch.uint8, device=device) for _ in range(4)]
    bf16 = torch.empty(count, dtype=torch.int16, device=device)
    _call("kvq_selftest_convert", first_bits & 0xFFFFFFFF, count, *(o.data_ptr() for o in outs),
          bf16.data_ptr(), _stream(stream, outs[0].device))
    return (*outs, bf16)
