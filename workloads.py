"""Seeded synthetic inputs for the quantized paged KV-cache workloads.

Shared by the tests, the benchmark and the smoke check.  This module only
draws random numbers and builds index structures (slot mappings, block
tables, request boundaries); it holds none of the method's arithmetic and
imports neither the CUDA binding nor the oracle.

Recipe (the pages print no dataset; these stand in for the prefill/decode
traffic they describe):
  * bf16 activations: float32 standard normals rounded to bf16.  Small cases
    use numpy's PCG64 (bit-identical on every machine); the two multi-GB cache
    fills can draw on the GPU with torch's seeded Philox generator.
  * decode-step outliers: each value independently scaled by 50 with p = 0.01
    (before the bf16 rounding).
  * slot mappings: distinct slots from a seeded permutation of the cache's
    slots, with a seeded set of positions replaced by -1 (padding).
  * gather batches: per-request lengths and start positions drawn uniformly;
    each request owns ceil((start + len) / block_size) blocks drawn without
    replacement from a seeded shuffle of all blocks; unused table entries -1.
  * workload k uses seed 1000 + k.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

NOPE_DIM = 512
ROPE_DIM = 64
NVFP4_DS_MLA_ENTRY = 352
FP8_DS_MLA_ENTRY = 656


# --------------------------------------------------------------------------
# primitive draws
# --------------------------------------------------------------------------

def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def normal_bf16(shape, seed: int, device="cpu", outlier_p: float = 0.0,
                outlier_scale: float = 50.0, rng: str = "numpy") -> torch.Tensor:
    """bf16 tensor of standard normals (optionally with sparse outliers).

    rng="numpy" draws on the host with PCG64 and copies to ``device``;
    rng="device" draws with torch's generator on ``device`` (fast for
    multi-GB fills; reproducible for a given device type)."""
    shape = tuple(int(s) for s in shape)
    if rng == "numpy":
        g = _rng(seed)
        x = g.standard_normal(shape, dtype=np.float32)
        if outlier_p > 0:
            x = np.where(g.random(shape, dtype=np.float32) < outlier_p,
                         x * np.float32(outlier_scale), x)
        return torch.from_numpy(x).to(torch.bfloat16).to(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if outlier_p > 0:
        u = torch.rand(shape, generator=gen, device=device, dtype=torch.float32)
        x = torch.where(u < outlier_p, x * outlier_scale, x)
    return x.to(torch.bfloat16)


def random_bytes(shape, seed: int) -> np.ndarray:
    """Uniform random uint8 array (cache pre-fill pattern)."""
    return _rng(seed).integers(0, 256, size=shape, dtype=np.uint8)


def nan_free_e4m3_bytes(a: np.ndarray) -> np.ndarray:
    """Replaces the two e4m3 NaN codes (0x7F, 0xFF) by 0x7E / 0xFE so that a
    random byte array holds finite e4m3 values only (in place; returned)."""
    a[a == 0x7F] = 0x7E
    a[a == 0xFF] = 0xFE
    return a


def slot_mapping(num_tokens: int, num_slots: int, num_pad: int, seed: int) -> np.ndarray:
    """num_tokens distinct slots drawn from range(num_slots), with num_pad
    seeded positions replaced by -1."""
    g = _rng(seed)
    if num_tokens > num_slots:
        raise ValueError("more tokens than slots")
    slots = g.permutation(num_slots)[:num_tokens].astype(np.int64)
    if num_pad:
        slots[g.choice(num_tokens, size=num_pad, replace=False)] = -1
    return slots


# --------------------------------------------------------------------------
# workload containers
# --------------------------------------------------------------------------

@dataclass
class WriteWorkload:
    """Inputs of one MLA cache write (nvfp4_ds_mla: 352 B, fp8_ds_mla: 656 B)."""
    name: str
    kv_c: torch.Tensor          # bf16 [T, 512]
    k_pe: torch.Tensor          # bf16 [T, 64]
    slot_mapping: torch.Tensor  # int64 [T], < 0 = padding
    num_blocks: int
    block_size: int
    entry_bytes: int

    @property
    def num_tokens(self) -> int:
        return int(self.slot_mapping.shape[0])

    @property
    def num_slots(self) -> int:
        return self.num_blocks * self.block_size


@dataclass
class GatherWorkload:
    """A cache fill plus one chunked-prefill gather over it."""
    name: str
    fill: WriteWorkload            # writes every slot of the cache
    block_table: torch.Tensor      # int32 [B, W], -1 = unused
    workspace_starts: torch.Tensor # int32 [B] (cu_seq_lens without its last entry)
    seq_starts: torch.Tensor       # int32 [B]
    seq_lens: list = field(default_factory=list)
    num_out_tokens: int = 0

    @property
    def batch_size(self) -> int:
        return int(self.seq_starts.shape[0])


@dataclass
class PerHeadWorkload:
    """Inputs of one per-head NVFP4 reshape_and_cache."""
    name: str
    key: torch.Tensor           # bf16 [T, H, D]
    value: torch.Tensor         # bf16 [T, H, D]
    slot_mapping: torch.Tensor  # int64 [T]
    num_pages: int
    block_size: int
    k_scale: float = 1.0
    v_scale: float = 1.0

    @property
    def num_tokens(self) -> int:
        return int(self.slot_mapping.shape[0])


@dataclass
class AttentionWorkload:
    """Sparse MLA attention (MQA form) of T decode tokens over a filled
    nvfp4_ds_mla cache."""
    name: str
    fill: WriteWorkload           # writes every slot of the cache
    q: torch.Tensor               # bf16 [T, H, 576]
    indices: torch.Tensor         # int32 [T, topk] global slots, -1 = unused
    softmax_scale: float

    @property
    def num_tokens(self) -> int:
        return int(self.q.shape[0])


@dataclass
class PrefillWorkload:
    """Dense prefill: the query tokens of each request attend to every
    position of its context, read through its block-table row."""
    name: str
    fill: WriteWorkload           # writes every slot of the cache
    q: torch.Tensor               # bf16 [T, H, 576]
    query_start: torch.Tensor     # int32 [B + 1]: request b owns query tokens [qs[b], qs[b+1])
    context_lens: torch.Tensor    # int32 [B]
    block_table: torch.Tensor     # int32 [B, W]
    softmax_scale: float
    max_query_len: int

    @property
    def num_tokens(self) -> int:
        return int(self.q.shape[0])


# --------------------------------------------------------------------------
# builders
# --------------------------------------------------------------------------

def make_write(name: str, num_tokens: int, num_blocks: int, block_size: int, num_pad: int,
               seed: int, device="cpu", entry_bytes: int = NVFP4_DS_MLA_ENTRY,
               outlier_p: float = 0.0, rng: str = "numpy", slots=None) -> WriteWorkload:
    """Write workload with distinct random slots (or the given slot array)."""
    if slots is None:
        slots = slot_mapping(num_tokens, num_blocks * block_size, num_pad, seed)
    kv_c = normal_bf16((num_tokens, NOPE_DIM), seed * 7 + 1, device, outlier_p=outlier_p, rng=rng)
    k_pe = normal_bf16((num_tokens, ROPE_DIM), seed * 7 + 2, device, rng=rng)
    return WriteWorkload(name, kv_c, k_pe, torch.from_numpy(np.asarray(slots, np.int64)).to(device),
                         num_blocks, block_size, entry_bytes)


def make_fill(name: str, num_blocks: int, block_size: int, seed: int, device="cpu",
              entry_bytes: int = NVFP4_DS_MLA_ENTRY, rng: str = "numpy") -> WriteWorkload:
    """A write of every slot of the cache, in a seeded shuffled order."""
    n = num_blocks * block_size
    slots = _rng(seed).permutation(n).astype(np.int64)
    return make_write(name, n, num_blocks, block_size, 0, seed, device, entry_bytes, rng=rng,
                      slots=slots)


def make_gather_batch(num_blocks: int, block_size: int, seq_lens, seq_starts, seed: int):
    """Block table, workspace starts and seq starts for requests with the
    given lengths and start positions; blocks are distinct and shuffled."""
    seq_lens = [int(x) for x in seq_lens]
    seq_starts = [int(x) for x in seq_starts]
    need = [-(-(s + n) // block_size) for s, n in zip(seq_starts, seq_lens)]
    if sum(need) > num_blocks:
        raise ValueError("batch needs more blocks than the cache has")
    width = max(max(need), 1)
    order = _rng(seed).permutation(num_blocks).astype(np.int32)
    table = np.full((len(seq_lens), width), -1, np.int32)
    pos = 0
    for b, k in enumerate(need):
        table[b, :k] = order[pos:pos + k]
        pos += k
    ws = np.zeros(len(seq_lens), np.int32)
    if len(seq_lens) > 1:
        ws[1:] = np.cumsum(seq_lens[:-1])
    return table, ws, np.asarray(seq_starts, np.int32), int(sum(seq_lens))


def make_gather(name: str, fill: WriteWorkload, seq_lens, seq_starts, seed: int,
                device="cpu") -> GatherWorkload:
    table, ws, starts, total = make_gather_batch(fill.num_blocks, fill.block_size, seq_lens,
                                                 seq_starts, seed)
    return GatherWorkload(name, fill, torch.from_numpy(table).to(device),
                          torch.from_numpy(ws).to(device), torch.from_numpy(starts).to(device),
                          list(int(x) for x in seq_lens), total)


def make_per_head(name: str, num_tokens: int, num_heads: int, head_size: int, num_pages: int,
                  block_size: int, num_pad: int, seed: int, device="cpu", k_scale: float = 1.0,
                  v_scale: float = 1.0, rng: str = "numpy") -> PerHeadWorkload:
    slots = slot_mapping(num_tokens, num_pages * block_size, num_pad, seed)
    key = normal_bf16((num_tokens, num_heads, head_size), seed * 7 + 3, device, rng=rng)
    value = normal_bf16((num_tokens, num_heads, head_size), seed * 7 + 4, device, rng=rng)
    return PerHeadWorkload(name, key, value, torch.from_numpy(slots).to(device), num_pages,
                           block_size, k_scale, v_scale)


def attention_indices(num_tokens: int, topk: int, num_slots: int, p_unused: float, seed: int) -> np.ndarray:
    """int32 [T, topk] slots drawn uniformly from the cache (a token's top-k
    positions land on scattered pages); entries set to -1 with p_unused."""
    g = _rng(seed)
    idx = g.integers(0, num_slots, size=(num_tokens, topk), dtype=np.int64).astype(np.int32)
    if p_unused > 0:
        idx[g.random((num_tokens, topk)) < p_unused] = -1
    return idx


def make_attention(name: str, num_tokens: int, num_heads: int, topk: int, num_blocks: int,
                   block_size: int, seed: int, device="cpu", p_unused: float = 0.0,
                   softmax_scale: float = 576 ** -0.5, q_scale: float = 1.0, fill: WriteWorkload = None,
                   rng: str = "numpy") -> AttentionWorkload:
    """Queries ~ q_scale * N(0, 1) in bf16 and top-k slot lists over a cache
    whose every slot is written (``fill``, or a fresh seeded fill)."""
    if fill is None:
        fill = make_fill(name + " fill", num_blocks, block_size, seed, device, rng=rng)
    q = normal_bf16((num_tokens, num_heads, NOPE_DIM + ROPE_DIM), seed * 7 + 5, device, rng=rng)
    if q_scale != 1.0:
        q = (q.float() * q_scale).to(torch.bfloat16)
    idx = attention_indices(num_tokens, topk, fill.num_slots, p_unused, seed * 7 + 6)
    return AttentionWorkload(name, fill, q, torch.from_numpy(idx).to(device), float(softmax_scale))


def make_prefill(name: str, context_lens, query_lens, num_heads: int, num_blocks: int, block_size: int,
                 seed: int, device="cpu", softmax_scale: float = 576 ** -0.5, fill: WriteWorkload = None,
                 rng: str = "numpy", block_table=None) -> PrefillWorkload:
    """Queries ~ N(0, 1) in bf16 for requests with the given query-token
    counts, each attending to its first context_lens[b] positions; each
    request owns distinct shuffled blocks (or the given block table) of a
    cache whose every slot is written (``fill``, or a fresh seeded fill)."""
    context_lens = [int(x) for x in context_lens]
    query_lens = [int(x) for x in query_lens]
    if fill is None:
        fill = make_fill(name + " fill", num_blocks, block_size, seed, device, rng=rng)
    if block_table is None:
        block_table = make_gather_batch(num_blocks, block_size, context_lens, [0] * len(context_lens), seed)[0]
    qs = np.zeros(len(query_lens) + 1, np.int32)
    qs[1:] = np.cumsum(query_lens)
    q = normal_bf16((int(qs[-1]), num_heads, NOPE_DIM + ROPE_DIM), seed * 7 + 5, device, rng=rng)
    return PrefillWorkload(name, fill, q, torch.from_numpy(qs).to(device),
                           torch.from_numpy(np.asarray(context_lens, np.int32)).to(device),
                           torch.as_tensor(np.asarray(block_table, np.int32)).to(device), float(softmax_scale),
                           max(query_lens) if query_lens else 0)


# --------------------------------------------------------------------------
# the five named workloads
# --------------------------------------------------------------------------

def smoke_write(device="cpu") -> WriteWorkload:
    """256 tokens into an 8 x 64 x 352 cache: the first 256 of a seeded
    permutation of its 512 slots, 16 of them set to -1."""
    return make_write("nvfp4_ds_mla write T=256 (8x64 cache, 16 pad)", 256, 8, 64, 16, 1001, device)


def smoke_gather(device="cpu") -> GatherWorkload:
    """Every slot of the 8 x 64 cache filled, then 2 requests with seq_starts
    {0, 17} and lengths {100, 120} gathered (220 rows)."""
    fill = make_fill("nvfp4_ds_mla fill 8x64", 8, 64, 1001, device)
    return make_gather("nvfp4_ds_mla gather B=2 T=220", fill, [100, 120], [0, 17], 1001, device)


def decode_write(device="cpu") -> WriteWorkload:
    """8192 decode tokens, 1% x50 outliers, into a 4096 x 64 x 352 cache;
    slots drawn from 262,144 free slots, 164 (2%) padding."""
    return make_write("nvfp4_ds_mla decode write T=8192 (4096x64 cache, 2% pad)", 8192, 4096, 64,
                      164, 1002, device, outlier_p=0.01)


def prefill_gather(device="cpu", rng: str | None = None) -> GatherWorkload:
    """65536 x 64 x 352 cache filled over all 4,194,304 slots, then 32
    requests with lengths U{4096..32768} and seq_starts U{1..4095}."""
    if rng is None:
        rng = "device" if str(device).startswith("cuda") else "numpy"
    g = _rng(1003)
    lens = g.integers(4096, 32768, size=32, endpoint=True)
    starts = g.integers(1, 4095, size=32, endpoint=True)
    fill = make_fill("nvfp4_ds_mla fill 65536x64 (4,194,304 tokens)", 65536, 64, 1003, device,
                     rng=rng)
    return make_gather("nvfp4_ds_mla gather B=32 len U[4k,32k]", fill, lens, starts, 1003, device)


def fp8_gather(device="cpu", rng: str | None = None) -> GatherWorkload:
    """32768 x 64 x 656 fp8_ds_mla cache filled over all 2,097,152 slots,
    then 16 requests of 16384 rows with seq_starts U{1..4095}."""
    if rng is None:
        rng = "device" if str(device).startswith("cuda") else "numpy"
    g = _rng(1004)
    starts = g.integers(1, 4095, size=16, endpoint=True)
    fill = make_fill("fp8_ds_mla fill 32768x64 (2,097,152 tokens)", 32768, 64, 1004, device,
                     entry_bytes=FP8_DS_MLA_ENTRY, rng=rng)
    return make_gather("fp8_ds_mla gather B=16 len 16384", fill, [16384] * 16, starts, 1004, device)


def per_head(device="cpu") -> PerHeadWorkload:
    """K, V bf16 [16384, 8, 128] into a 16384 x 2 x 16 x 8 x 72 cache; 16384
    distinct slots of 262,144; scales 1.0."""
    return make_per_head("per-head nvfp4 T=16384 H=8 D=128 (16384 pages x 16)", 16384, 8, 128,
                         16384, 16, 0, 1005, device)


def sparse_attention(device="cpu", fill: WriteWorkload = None) -> AttentionWorkload:
    """Sparse MLA decode: 4096 tokens x 128 heads, top-2048 slots each (10 %
    unused) drawn over the given cache fill (else a fresh 65536 x 64
    nvfp4_ds_mla fill), softmax scale 576^-0.5."""
    return make_attention("sparse MLA attention T=4096 H=128 top-2048", 4096, 128, 2048, 65536, 64, 1006,
                          device, p_unused=0.1, fill=fill,
                          rng="device" if str(device).startswith("cuda") else "numpy")


def prefill_attention(gather: GatherWorkload, device="cpu", query_len: int = 16) -> PrefillWorkload:
    """Dense prefill over the prefill gather's cache and batch: each of its 32
    requests attends with ``query_len`` new tokens x 128 heads to its whole
    context up to the end of its gathered range (seq_start + length, 4k-36k
    positions) through the same block table."""
    ctx = [int(s) + n for s, n in zip(host(gather.seq_starts), gather.seq_lens)]
    return make_prefill(f"dense prefill B={len(ctx)} q={query_len} H=128 over contexts of 4k-36k", ctx,
                        [query_len] * len(ctx), 128, gather.fill.num_blocks, gather.fill.block_size, 1007, device,
                        fill=gather.fill, rng="device" if str(device).startswith("cuda") else "numpy",
                        block_table=host(gather.block_table))


# --------------------------------------------------------------------------
# host views for the oracle
# --------------------------------------------------------------------------

def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """numpy uint16 bit patterns of a bf16 tensor (copied to the host)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy()
