"""CPU oracle for the quantized paged KV-cache write and gather-upconvert path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` import this package.  It wraps the plain
C library built from ``oracle/kvq_oracle.c`` (see that file for the citations
of every step) with numpy marshalling; no arithmetic of the method lives in
this Python file.

bf16 tensors are passed as ``numpy.uint16`` bit patterns.  Token-range ops
accept ``threads``: the range is cut into contiguous chunks that run the same
single-threaded C function side by side (ctypes releases the GIL), which is
only valid because distinct tokens write distinct slots.
"""
from __future__ import annotations

import ctypes
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import build as _build

_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_U32 = ctypes.c_uint32
_F32 = ctypes.c_float

_SIGNATURES = {
    "kvqo_e4m3_value": (ctypes.c_double, [ctypes.c_uint8]),
    "kvqo_e2m1_value": (ctypes.c_double, [ctypes.c_uint8]),
    "kvqo_bf16_value": (ctypes.c_float, [ctypes.c_uint16]),
    "kvqo_e4m3_rn_sat": (ctypes.c_uint8, [_F32]),
    "kvqo_e2m1_rn_sat": (ctypes.c_uint8, [_F32]),
    "kvqo_bf16_rn": (ctypes.c_uint16, [_F32]),
    "kvqo_encode_bits_range": (None, [_U32, _I64, _P, _P]),
    "kvqo_bf16_rn_bits_range": (None, [_U32, _I64, _P]),
    "kvqo_e4m3_rn_sat_array": (None, [_P, _I64, _P]),
    "kvqo_e2m1_rn_sat_array": (None, [_P, _I64, _P]),
    "kvqo_bf16_rn_array": (None, [_P, _I64, _P]),
    "kvqo_nvfp4_ds_mla_entry_bytes": (_I32, []),
    "kvqo_fp8_ds_mla_entry_bytes": (_I32, []),
    "kvqo_nvfp4_full_dim": (_I32, [_I32]),
    "kvqo_nvfp4_data_dim": (_I32, [_I32]),
    "kvqo_nvfp4_scale_dim": (_I32, [_I32]),
    "kvqo_write_nvfp4_ds_mla": (_I64, [_P, _I64, _P, _I64, _P, _I64, _I64, _P, _I64, _I32, _I64, _I64]),
    "kvqo_write_fp8_ds_mla": (_I64, [_P, _I64, _P, _I64, _P, _I64, _I64, _P, _I64, _I32, _I64, _I64]),
    "kvqo_gather_nvfp4_ds_mla": (_I64, [_P, _I64, _I32, _I64, _I64, _P, _I64, _I64, _P, _I64, _I32,
                                        _P, _P, _I32, _P, _I64]),
    "kvqo_gather_fp8_ds_mla": (_I64, [_P, _I64, _I32, _I64, _I64, _P, _I64, _I64, _P, _I64, _I32,
                                      _P, _P, _I32, _P, _I64]),
    "kvqo_reshape_and_cache_nvfp4": (_I64, [_P, _P, _I64, _I64, _I64, _I64, _P, _I64, _I64, _I32, _I32,
                                            _P, _I64, _I32, _F32, _F32, _I32]),
    "kvqo_dequant_nvfp4_per_head": (_I64, [_P, _I64, _I32, _I32, _I32, _P, _I64, _I64, _F32, _F32, _I32,
                                           _P, _P]),
    "kvqo_req_index_to_global_slot": (_I64, [_P, _P, _I64, _I32, _P, _I64, _I32, _I32, _I32, _I64, _P]),
    "kvqo_sparse_mla_attention_nvfp4_ds_mla": (_I64, [_P, _I64, _I64, _I64, _I64, _I32, _P, _I64, _I32,
                                                      _P, _I64, _I32, _I64, _I64, ctypes.c_double,
                                                      _P, _I64, _I64, _P, _I64]),
    "kvqo_sparse_mla_attention_fp8_ds_mla": (_I64, [_P, _I64, _I64, _I64, _I64, _I32, _P, _I64, _I32,
                                                    _P, _I64, _I32, _I64, _I64, ctypes.c_double,
                                                    _P, _I64, _I64, _P, _I64]),
    "kvqo_prefill_mla_attention_nvfp4_ds_mla": (_I64, [_P, _I64, _I64, _I32, _P, _P, _P, _I64, _I32, _I64, _I64,
                                                       _P, _I64, _I32, _I64, _I64, ctypes.c_double,
                                                       _P, _I64, _I64, _P, _I64]),
    "kvqo_prefill_mla_attention_fp8_ds_mla": (_I64, [_P, _I64, _I64, _I32, _P, _P, _P, _I64, _I32, _I64, _I64,
                                                     _P, _I64, _I32, _I64, _I64, ctypes.c_double,
                                                     _P, _I64, _I64, _P, _I64]),
    "kvqo_decode_fp8_ds_mla_entry": (None, [_P, _P]),
    "kvqo_decode_nvfp4_ds_mla_entry": (None, [_P, _P]),
}


def lib():
    """Loads (building first if needed) the oracle library."""
    global _lib
    if _lib is None:
        path = _build.build()
        handle = ctypes.CDLL(path)
        for name, (restype, argtypes) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = restype
            fn.argtypes = argtypes
        _lib = handle
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _run_chunks(fn, n: int, threads: int):
    """Calls fn(begin, end) over [0, n) in contiguous chunks; sums results."""
    threads = max(1, min(int(threads), n)) if n > 0 else 1
    if threads == 1:
        return fn(0, n)
    bounds = np.linspace(0, n, threads + 1).astype(np.int64)
    with ThreadPoolExecutor(max_workers=threads) as pool:
        futures = [pool.submit(fn, int(bounds[i]), int(bounds[i + 1])) for i in range(threads)]
        return sum(f.result() for f in futures)


def default_threads() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


# --------------------------------------------------------------------------
# scalar / array converters
# --------------------------------------------------------------------------

def e4m3_value(code: int) -> float:
    return lib().kvqo_e4m3_value(code)


def e2m1_value(nibble: int) -> float:
    return lib().kvqo_e2m1_value(nibble)


def e4m3_rn_sat(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().kvqo_e4m3_rn_sat_array(_ptr(x), x.size, _ptr(out))
    return out


def e2m1_rn_sat(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().kvqo_e2m1_rn_sat_array(_ptr(x), x.size, _ptr(out))
    return out


def bf16_rn(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().kvqo_bf16_rn_array(_ptr(x), x.size, _ptr(out))
    return out


def encode_bits_range(first_bits: int, count: int, threads: int = 1):
    """e4m3 and e2m1 codes of the float32 bit patterns first..first+count-1."""
    e4m3 = np.empty(count, np.uint8)
    e2m1 = np.empty(count, np.uint8)
    base4, base2 = e4m3.ctypes.data, e2m1.ctypes.data

    def run(b, e):
        lib().kvqo_encode_bits_range((first_bits + b) & 0xFFFFFFFF, e - b, base4 + b, base2 + b)
        return 0

    _run_chunks(run, count, threads)
    return e4m3, e2m1


def bf16_rn_bits_range(first_bits: int, count: int, threads: int = 1) -> np.ndarray:
    out = np.empty(count, np.uint16)
    base = out.ctypes.data

    def run(b, e):
        lib().kvqo_bf16_rn_bits_range((first_bits + b) & 0xFFFFFFFF, e - b, base + 2 * b)
        return 0

    _run_chunks(run, count, threads)
    return out


# --------------------------------------------------------------------------
# format constants
# --------------------------------------------------------------------------

def nvfp4_ds_mla_entry_bytes() -> int:
    return lib().kvqo_nvfp4_ds_mla_entry_bytes()


def fp8_ds_mla_entry_bytes() -> int:
    return lib().kvqo_fp8_ds_mla_entry_bytes()


def nvfp4_full_dim(head_size: int) -> int:
    return lib().kvqo_nvfp4_full_dim(head_size)


def nvfp4_data_dim(full_dim: int) -> int:
    return lib().kvqo_nvfp4_data_dim(full_dim)


def nvfp4_scale_dim(full_dim: int) -> int:
    return lib().kvqo_nvfp4_scale_dim(full_dim)


# --------------------------------------------------------------------------
# operations
# --------------------------------------------------------------------------

def _rows_of(a: np.ndarray) -> int:
    return a.strides[0] // a.itemsize


def _check_bf16_rows(name: str, a: np.ndarray, width: int):
    if a.dtype != np.uint16 or a.ndim != 2 or a.shape[1] < width or a.strides[1] != 2:
        raise ValueError(f"{name}: expected uint16 [T, >={width}] rows with unit inner stride")


def _cache_geometry(cache: np.ndarray, entry_bytes: int):
    """(num_blocks, block_size, block_stride, entry_stride) of a uint8 cache
    shaped [num_blocks, block_size, >= entry_bytes] with unit inner stride."""
    if cache.dtype != np.uint8 or cache.ndim != 3 or cache.shape[2] < entry_bytes or cache.strides[2] != 1:
        raise ValueError(f"cache: expected uint8 [num_blocks, block_size, >={entry_bytes}]")
    return cache.shape[0], cache.shape[1], cache.strides[0], cache.strides[1]


def _write(fn_name, entry_bytes, kv_c, k_pe, slot_mapping, cache, threads):
    _check_bf16_rows("kv_c", kv_c, 512)
    _check_bf16_rows("k_pe", k_pe, 64)
    slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    nb, bs, bstride, estride = _cache_geometry(cache, entry_bytes)
    fn = getattr(lib(), fn_name)
    T = slot_mapping.shape[0]
    if kv_c.shape[0] < T or k_pe.shape[0] < T:
        raise ValueError("fewer kv_c / k_pe rows than slots")

    def run(b, e):
        return fn(_ptr(kv_c), _rows_of(kv_c), _ptr(k_pe), _rows_of(k_pe), _ptr(slot_mapping), b, e,
                  _ptr(cache), nb, bs, bstride, estride)

    return _run_chunks(run, T, threads)


def write_nvfp4_ds_mla(kv_c, k_pe, slot_mapping, cache, threads: int = 1) -> int:
    """In-place oracle write of the 352-byte nvfp4_ds_mla entries; returns the
    number of out-of-range slots skipped."""
    return _write("kvqo_write_nvfp4_ds_mla", 352, kv_c, k_pe, slot_mapping, cache, threads)


def write_fp8_ds_mla(kv_c, k_pe, slot_mapping, cache, threads: int = 1) -> int:
    """In-place oracle write of the 656-byte fp8_ds_mla entries."""
    return _write("kvqo_write_fp8_ds_mla", 656, kv_c, k_pe, slot_mapping, cache, threads)


def _gather(fn_name, entry_bytes, cache, block_table, workspace_starts, seq_starts,
            num_out_tokens, rows, dst, threads):
    nb, bs, bstride, estride = _cache_geometry(cache, entry_bytes)
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    workspace_starts = np.ascontiguousarray(workspace_starts, dtype=np.int32)
    seq_starts = np.ascontiguousarray(seq_starts, dtype=np.int32)
    B = seq_starts.shape[0]
    if workspace_starts.shape[0] < B or block_table.shape[0] < B:
        raise ValueError("workspace_starts / block_table have fewer than batch_size rows")
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = num_out_tokens if rows is None else rows.shape[0]
    if dst is None:
        dst = np.zeros((n, 576), np.uint16)
    _check_bf16_rows("dst", dst, 576)
    fn = getattr(lib(), fn_name)
    W = block_table.shape[1]

    def run(b, e):
        r = np.arange(b, e, dtype=np.int64) if rows is None else rows[b:e]
        return fn(_ptr(cache), nb, bs, bstride, estride, dst.ctypes.data + b * dst.strides[0],
                  _rows_of(dst), num_out_tokens, _ptr(block_table), W, W, _ptr(workspace_starts),
                  _ptr(seq_starts), B, r.ctypes.data, e - b)

    skipped = _run_chunks(run, n, threads)
    return dst, skipped


def gather_nvfp4_ds_mla(cache, block_table, workspace_starts, seq_starts, num_out_tokens,
                        rows=None, dst=None, threads: int = 1):
    """Oracle gather-upconvert of nvfp4_ds_mla pages; returns (dst uint16
    [n, 576], rows skipped).  ``rows`` selects workspace rows (dst row i is
    workspace row rows[i]); ``dst`` may be passed to keep untouched rows."""
    return _gather("kvqo_gather_nvfp4_ds_mla", 352, cache, block_table, workspace_starts,
                   seq_starts, num_out_tokens, rows, dst, threads)


def gather_fp8_ds_mla(cache, block_table, workspace_starts, seq_starts, num_out_tokens,
                      rows=None, dst=None, threads: int = 1):
    """Oracle gather-upconvert of fp8_ds_mla pages (see gather_nvfp4_ds_mla)."""
    return _gather("kvqo_gather_fp8_ds_mla", 656, cache, block_table, workspace_starts,
                   seq_starts, num_out_tokens, rows, dst, threads)


def _check_khd(name, a):
    if a.dtype != np.uint16 or a.ndim != 3 or a.strides[2] != 2:
        raise ValueError(f"{name}: expected uint16 [T, H, D] with unit inner stride")


LAYOUTS = {"NHD": 0, "HND": 1}


def _per_head_geometry(cache, H, D, layout):
    """(num_pages, block_size) of a contiguous per-head cache: uint8
    [P, 2, block_size, H, full_dim] for NHD, [P, 2, H, block_size, full_dim]
    for HND."""
    if layout not in LAYOUTS:
        raise ValueError("layout must be 'NHD' or 'HND'")
    if cache.dtype != np.uint8 or cache.ndim != 5 or not cache.flags.c_contiguous:
        raise ValueError("cache: expected a contiguous uint8 5-d per-head cache")
    P, two, d2, d3, fd = cache.shape
    bs, Hc = (d2, d3) if layout == "NHD" else (d3, d2)
    if two != 2 or Hc != H or fd != nvfp4_full_dim(D):
        raise ValueError("cache shape does not match key / value")
    return P, bs


def reshape_and_cache_nvfp4(key, value, slot_mapping, cache, k_scale: float = 1.0,
                            v_scale: float = 1.0, threads: int = 1, layout: str = "NHD") -> int:
    """In-place oracle write of the per-head NVFP4 cache (uint8
    [num_pages, 2, block_size, H, full_dim] for NHD, [.., H, block_size, ..]
    for HND); returns out-of-range slots."""
    _check_khd("key", key)
    _check_khd("value", value)
    T, H, D = key.shape
    if value.shape != key.shape:
        raise ValueError("key / value shapes differ")
    P, bs = _per_head_geometry(cache, H, D, layout)
    slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    fn = lib().kvqo_reshape_and_cache_nvfp4

    def run(b, e):
        return fn(_ptr(key), _ptr(value), key.strides[0] // 2, key.strides[1] // 2,
                  value.strides[0] // 2, value.strides[1] // 2, _ptr(slot_mapping), b, e,
                  H, D, _ptr(cache), P, bs, k_scale, v_scale, LAYOUTS[layout])

    return _run_chunks(run, slot_mapping.shape[0], threads)


def dequant_nvfp4_per_head(cache, slot_mapping, num_heads: int, head_size: int,
                           k_scale: float = 1.0, v_scale: float = 1.0,
                           key_out=None, value_out=None, threads: int = 1, layout: str = "NHD"):
    """Reads the per-head cache back at slot_mapping into bf16 [T, H, D]."""
    P, bs = _per_head_geometry(cache, num_heads, head_size, layout)
    slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T = slot_mapping.shape[0]
    if key_out is None:
        key_out = np.zeros((T, num_heads, head_size), np.uint16)
    if value_out is None:
        value_out = np.zeros((T, num_heads, head_size), np.uint16)
    fn = lib().kvqo_dequant_nvfp4_per_head

    def run(b, e):
        return fn(_ptr(cache), P, bs, num_heads, head_size, _ptr(slot_mapping), b, e,
                  k_scale, v_scale, LAYOUTS[layout], _ptr(key_out), _ptr(value_out))

    skipped = _run_chunks(run, T, threads)
    return key_out, value_out, skipped


def req_index_to_global_slot(req_id, token_indices, block_table, block_size: int, num_blocks: int):
    """Oracle sparse-decode index conversion; returns (int32 [N, topk], skipped)."""
    req_id = np.ascontiguousarray(req_id, dtype=np.int32)
    token_indices = np.ascontiguousarray(token_indices, dtype=np.int32)
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    N, topk = token_indices.shape
    if req_id.shape[0] != N:
        raise ValueError("req_id and token_indices lengths differ")
    out = np.empty((N, topk), np.int32)
    skipped = lib().kvqo_req_index_to_global_slot(
        _ptr(req_id), _ptr(token_indices), N, topk, _ptr(block_table), block_table.shape[1],
        block_table.shape[1], block_table.shape[0], block_size, num_blocks, _ptr(out))
    return out, skipped


def sparse_mla_attention_nvfp4_ds_mla(q, indices, cache, softmax_scale: float, threads: int = 1):
    """Oracle sparse MLA attention (MQA form) of q uint16 bf16 bits [T, H, 576]
    over the global slots indices int32 [T, topk] of the nvfp4_ds_mla cache;
    returns (o float64 [T, H, 512], lse float64 [T, H], slots skipped)."""
    return _attention("kvqo_sparse_mla_attention_nvfp4_ds_mla", 352, q, indices, cache, softmax_scale, threads)


def sparse_mla_attention_fp8_ds_mla(q, indices, cache, softmax_scale: float, threads: int = 1):
    """The same over the 656-byte fp8_ds_mla cache."""
    return _attention("kvqo_sparse_mla_attention_fp8_ds_mla", 656, q, indices, cache, softmax_scale, threads)


def _attention(fn_name, entry_bytes, q, indices, cache, softmax_scale, threads):
    if q.dtype != np.uint16 or q.ndim != 3 or q.shape[2] != 576 or q.strides[2] != 2:
        raise ValueError("q: expected uint16 [T, H, 576] with unit inner stride")
    indices = np.ascontiguousarray(indices, dtype=np.int32)
    T, H = q.shape[0], q.shape[1]
    if indices.ndim != 2 or indices.shape[0] != T:
        raise ValueError("indices: expected int32 [T, topk]")
    nb, bs, bstride, estride = _cache_geometry(cache, entry_bytes)
    out = np.zeros((T, H, 512), np.float64)
    lse = np.zeros((T, H), np.float64)
    fn = getattr(lib(), fn_name)

    def run(b, e):
        r = fn(_ptr(q), q.strides[0] // 2, q.strides[1] // 2, b, e, H, _ptr(indices), indices.shape[1],
               indices.shape[1], _ptr(cache), nb, bs, bstride, estride, float(softmax_scale),
               _ptr(out), H * 512, 512, _ptr(lse), H)
        if r < 0:
            raise MemoryError("oracle attention: scratch allocation failed")
        return r

    skipped = _run_chunks(run, T, threads)
    return out, lse, skipped


def prefill_mla_attention_nvfp4_ds_mla(q, query_start, context_lens, block_table, cache, softmax_scale: float,
                                       threads: int = 1):
    """Oracle dense prefill over the nvfp4_ds_mla cache: q uint16 bf16 bits [T,
    H, 576]; request b's query tokens [query_start[b], query_start[b+1])
    attend to its context positions [0, context_lens[b]) through block_table
    int32 [B, W]; returns (o float64 [T, H, 512], lse float64 [T, H],
    positions skipped)."""
    return _prefill("kvqo_prefill_mla_attention_nvfp4_ds_mla", 352, q, query_start, context_lens, block_table,
                    cache, softmax_scale, threads)


def prefill_mla_attention_fp8_ds_mla(q, query_start, context_lens, block_table, cache, softmax_scale: float,
                                     threads: int = 1):
    """The same over the 656-byte fp8_ds_mla cache."""
    return _prefill("kvqo_prefill_mla_attention_fp8_ds_mla", 656, q, query_start, context_lens, block_table,
                    cache, softmax_scale, threads)


def _prefill(fn_name, entry_bytes, q, query_start, context_lens, block_table, cache, softmax_scale, threads):
    if q.dtype != np.uint16 or q.ndim != 3 or q.shape[2] != 576 or q.strides[2] != 2:
        raise ValueError("q: expected uint16 [T, H, 576] with unit inner stride")
    query_start = np.ascontiguousarray(query_start, dtype=np.int32)
    context_lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    B = context_lens.shape[0]
    if query_start.shape != (B + 1,) or block_table.ndim != 2 or block_table.shape[0] != B:
        raise ValueError("query_start [B + 1], context_lens [B] and block_table [B, W] disagree")
    T, H = q.shape[0], q.shape[1]
    if query_start[0] < 0 or query_start[-1] > T or np.any(np.diff(query_start) < 0):
        raise ValueError("query_start must be non-decreasing within [0, T]")
    nb, bs, bstride, estride = _cache_geometry(cache, entry_bytes)
    out = np.zeros((T, H, 512), np.float64)
    lse = np.zeros((T, H), np.float64)
    fn = getattr(lib(), fn_name)

    def run(b, e):
        r = fn(_ptr(q), q.strides[0] // 2, q.strides[1] // 2, H, _ptr(query_start), _ptr(context_lens),
               _ptr(block_table), block_table.shape[1], block_table.shape[1], b, e, _ptr(cache), nb, bs, bstride,
               estride, float(softmax_scale), _ptr(out), H * 512, 512, _ptr(lse), H)
        if r < 0:
            raise MemoryError("oracle prefill attention: scratch allocation failed")
        return r

    skipped = _run_chunks(run, B, threads)
    return out, lse, skipped


def decode_fp8_ds_mla_entry(entry) -> np.ndarray:
    """The 576 bf16 values (as float64) one 656-byte fp8_ds_mla entry upconverts to."""
    entry = np.ascontiguousarray(entry, dtype=np.uint8)
    if entry.shape != (656,):
        raise ValueError("entry must be 656 bytes")
    out = np.empty(576, np.float64)
    lib().kvqo_decode_fp8_ds_mla_entry(_ptr(entry), _ptr(out))
    return out


def decode_nvfp4_ds_mla_entry(entry) -> np.ndarray:
    """The 576 values (as float64) one 352-byte entry decodes to."""
    entry = np.ascontiguousarray(entry, dtype=np.uint8)
    if entry.shape != (352,):
        raise ValueError("entry must be 352 bytes")
    out = np.empty(576, np.float64)
    lib().kvqo_decode_nvfp4_ds_mla_entry(_ptr(entry), _ptr(out))
    return out
