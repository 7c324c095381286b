"""GPU parity: every CUDA entry point against the CPU oracle, element by
element, on the same seeded inputs.  Integer / byte outputs (cache bytes) and
the bf16 gathers (exact or single-rounding results) must match bit for bit.

Small cases cover several CTAs and ragged tails plus edge cases (padding,
out-of-range indices, zero-length requests, padded strides, extreme values);
the full-size cases run the workloads the benchmark times, completely.
"""
import numpy as np
import pytest
import torch

import independent as ind
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


@pytest.fixture(scope="module")
def threads(oracle_mod):
    return oracle_mod.default_threads()


def dev(x):
    return x.to(DEV) if isinstance(x, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def finite_bf16_bits(shape, seed):
    """Random finite bf16 bit patterns over the whole exponent range (zeros,
    subnormals, huge values, both signs)."""
    b = wl.random_bytes(tuple(shape) + (2,), seed).view(np.uint16).reshape(shape)
    exp_all_ones = (b & 0x7F80) == 0x7F80
    b[exp_all_ones] &= 0xBFFF            # clear an exponent bit: finite
    return b


def bits_to_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


# --------------------------------------------------------------------------
# device converters, exhaustively over the exponent window that matters
# --------------------------------------------------------------------------

def test_device_converters_match_oracle_exhaustively(kvq, oracle_mod, threads):
    """All 2^32 float32 bit patterns through the device e4m3 / e2m1 / bf16
    converters (both lanes of the packed conversions) against the oracle.
    NaN inputs are outside the ops' contract; e4m3 must keep them NaN."""
    chunk = 1 << 26
    for first in range(0, 1 << 32, chunk):
        e4l, e4h, e2l, e2h, bf = (t.cpu().numpy() for t in kvq.kvq_selftest_convert(first, chunk))
        o4, o2 = oracle_mod.encode_bits_range(first, chunk, threads=threads)
        ob = oracle_mod.bf16_rn_bits_range(first, chunk, threads=threads)
        f = np.arange(first, first + chunk, dtype=np.uint64).astype(np.uint32).view(np.float32)
        nan = np.isnan(f)
        if not nan.any():
            ok = (np.array_equal(e4l, o4) and np.array_equal(e4h, o4) and np.array_equal(e2l, o2)
                  and np.array_equal(e2h, o2) and np.array_equal(bf.view(np.uint16), ob))
        else:
            keep = ~nan
            ok = (np.array_equal(e4l[keep], o4[keep]) and np.array_equal(e4h[keep], o4[keep])
                  and np.array_equal(e2l[keep], o2[keep]) and np.array_equal(e2h[keep], o2[keep])
                  and np.array_equal(bf.view(np.uint16)[keep], ob[keep])
                  and np.all((e4l[nan] & 0x7F) == 0x7F) and np.all((e4h[nan] & 0x7F) == 0x7F))
        assert ok, f"converter mismatch in patterns [{first:#x}, {first + chunk:#x})"


# --------------------------------------------------------------------------
# nvfp4_ds_mla / fp8_ds_mla writes
# --------------------------------------------------------------------------

def run_write(kvq, oracle_mod, w, entry, init_seed=3, pad_entry=0, pad_block=0, kv_view=False,
              threads=1, status_expected=0, narrow_rows=False):
    """GPU vs oracle write into a pre-filled cache with optional padded
    entries / blocks; returns the GPU cache (host)."""
    es = entry + pad_entry
    buf0 = wl.random_bytes((w.num_blocks, w.block_size + pad_block, es), init_seed)
    kv_bits, pe_bits = wl.bf16_bits(w.kv_c), wl.bf16_bits(w.k_pe)
    slots = wl.host(w.slot_mapping)
    if kv_view:            # kv_c and k_pe as column slices of one [T, 576] tensor
        both = torch.cat([w.kv_c, w.k_pe], dim=1).to(DEV)
        kv_c, k_pe = both[:, :512], both[:, 512:]
    elif narrow_rows:      # rows 16-byte but not 32-byte aligned: the two-access path
        buf = torch.zeros((w.num_tokens, 600), dtype=torch.bfloat16, device=DEV)
        buf[:, 8:520] = w.kv_c.to(DEV)
        buf[:, 528:592] = w.k_pe.to(DEV)
        kv_c, k_pe = buf[:, 8:520], buf[:, 528:592]
    else:
        kv_c, k_pe = dev(w.kv_c), dev(w.k_pe)
    gbuf = dev(buf0.copy())
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    fn = kvq.kvq_write_nvfp4_ds_mla if entry == 352 else kvq.kvq_write_fp8_ds_mla
    fn(kv_c, k_pe, gbuf[:, :w.block_size, :], dev(slots), status=status)
    want = buf0.copy()
    ofn = oracle_mod.write_nvfp4_ds_mla if entry == 352 else oracle_mod.write_fp8_ds_mla
    ofn(kv_bits, pe_bits, slots, want[:, :w.block_size, :entry], threads=threads)
    got = gbuf.cpu().numpy()
    assert int(status.item()) == status_expected
    np.testing.assert_array_equal(got, want)
    return got


WRITE_CASES = [
    ("smoke T=256", lambda: wl.smoke_write(), {}),
    ("decode T=8192 outliers", lambda: wl.decode_write(), {}),
    ("single token", lambda: wl.make_write("t1", 1, 1, 64, 0, 61), {}),
    ("ragged T=37", lambda: wl.make_write("t37", 37, 2, 64, 5, 62), {}),
    ("all padding", lambda: wl.make_write("pad", 40, 1, 64, 40, 63), {}),
    ("block_size 1", lambda: wl.make_write("bs1", 250, 300, 1, 3, 64), {}),
    ("block_size 16 padded strides", lambda: wl.make_write("bs16", 333, 40, 16, 9, 65),
     dict(pad_entry=16, pad_block=3)),
    ("kv_c / k_pe slices of one tensor", lambda: wl.make_write("view", 129, 4, 64, 2, 66),
     dict(kv_view=True)),
    ("block_size 7", lambda: wl.make_write("bs7", 300, 50, 7, 5, 67), {}),
    ("16-byte aligned rows", lambda: wl.make_write("narrow", 77, 4, 64, 3, 69), dict(narrow_rows=True)),
    ("4-token warps, ragged T=65573", lambda: wl.make_write("big", 65573, 2048, 64, 300, 70), {}),
    ("4-token warps, 16-byte aligned rows", lambda: wl.make_write("bign", 65540, 1100, 64, 17, 71),
     dict(narrow_rows=True)),
    ("block_size 33", lambda: wl.make_write("bs33", 301, 12, 33, 6, 68), {}),
]


@pytest.mark.parametrize("entry", [352, 656])
@pytest.mark.parametrize("name,make,kw", WRITE_CASES, ids=[c[0] for c in WRITE_CASES])
def test_write_parity(kvq, oracle_mod, threads, entry, name, make, kw):
    run_write(kvq, oracle_mod, make(), entry, threads=threads, **kw)


@pytest.mark.parametrize("entry", [352, 656])
def test_write_parity_extreme_values(kvq, oracle_mod, entry):
    """Random finite bf16 bit patterns (subnormals, zeros, huge values), plus
    all-zero and negative-zero groups and tiles."""
    T = 300
    kv = finite_bf16_bits((T, 512), 71)
    pe = finite_bf16_bits((T, 64), 72)
    kv[5, :] = 0
    kv[6, :] = 0x8000
    kv[7, :128] = 0x0001                       # smallest subnormal
    kv[8, 16:32] = 0x7F7F                      # largest finite
    slots = wl.slot_mapping(T, 8 * 64, 7, 73)
    w = wl.WriteWorkload("extreme", bits_to_bf16(kv), bits_to_bf16(pe), torch.from_numpy(slots), 8, 64, entry)
    run_write(kvq, oracle_mod, w, entry)


@pytest.mark.parametrize("base", [1.0, 1.5, 2.0 ** -7, 1.25 * 2.0 ** 9, 2.0 ** -64, 1.5 * 2.0 ** -65, 2.0 ** -100])
def test_fp8_write_quotients_on_e4m3_ties(kvq, oracle_mod, base):
    """fp8_ds_mla tiles whose values divide by the tile scale exactly onto
    e4m3 rounding ties (and exact codes): the quotient must be the exact one
    for round-to-nearest-even to pick the even code."""
    g = np.random.Generator(np.random.PCG64(171))
    mags = ind.e4m3_table()[:127]
    mids = (mags[:-1] + mags[1:]) / 2
    T = 48
    x = np.zeros((T, 512))
    for t in range(T):
        for j in range(4):
            vals = g.choice(np.concatenate([mids, mags]), 128) * g.choice([-1.0, 1.0], 128)
            vals[g.integers(0, 128)] = 448.0            # sets amax = 448 * base, so s = base
            x[t, 128 * j:128 * (j + 1)] = vals * base
    xb = ind.torch_bf16_bits(torch.from_numpy(x.astype(np.float32)))
    assert np.array_equal(ind.bf16_to_f32(xb).astype(np.float64), x)     # exact in bf16
    pe = finite_bf16_bits((T, 64), 172)
    w = wl.WriteWorkload("ties", bits_to_bf16(xb), bits_to_bf16(pe),
                         torch.from_numpy(np.arange(T, dtype=np.int64)), 1, 64, 656)
    run_write(kvq, oracle_mod, w, 656)


@pytest.mark.parametrize("entry", [352, 656])
def test_write_out_of_range_slots_are_skipped_and_reported(kvq, oracle_mod, entry):
    w = wl.make_write("oob", 100, 2, 64, 4, 74)
    slots = wl.host(w.slot_mapping).copy()
    slots[[3, 50, 99]] = [128, 10 ** 12, 129]
    w.slot_mapping = torch.from_numpy(slots)
    run_write(kvq, oracle_mod, w, entry, status_expected=kvq.STATUS_BAD_INDEX)


def test_write_prefill_fill_full_size(kvq, oracle_mod, threads):
    """The 65536 x 64 x 352 cache written over all 4,194,304 slots."""
    g = wl.prefill_gather(DEV)
    w = g.fill
    cache = torch.zeros((w.num_blocks, w.block_size, 352), dtype=torch.uint8, device=DEV)
    kvq.kvq_write_nvfp4_ds_mla(w.kv_c, w.k_pe, cache, w.slot_mapping)
    want = np.zeros((w.num_blocks, w.block_size, 352), np.uint8)
    oracle_mod.write_nvfp4_ds_mla(wl.bf16_bits(w.kv_c), wl.bf16_bits(w.k_pe), wl.host(w.slot_mapping),
                                  want, threads=threads)
    got = cache.cpu().numpy()
    assert np.array_equal(got, want), f"{int((got != want).sum())} bytes differ"


# --------------------------------------------------------------------------
# gathers
# --------------------------------------------------------------------------

def run_gather(kvq, oracle_mod, entry, cache_host, table, ws, starts, T, batch_size=None,
               dst_pad=0, pad_entry=0, pad_block=0, status_expected=0, threads=1, dst_offset=0):
    nb, bs, _ = cache_host.shape
    buf = np.zeros((nb, bs + pad_block, entry + pad_entry), np.uint8)
    buf[:, :bs, :entry] = cache_host
    gbuf = dev(buf)
    dst = torch.full((T, 576 + dst_pad + dst_offset), -7.0, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    fn = kvq.kvq_gather_upconvert_nvfp4_ds_mla if entry == 352 else kvq.kvq_gather_upconvert_fp8_ds_mla
    view = dst[:, dst_offset:dst_offset + 576] if (dst_pad or dst_offset) else dst
    fn(gbuf[:, :bs, :], view, dev(table), dev(ws), dev(starts), batch_size=batch_size, status=status)
    dst = dst[:, dst_offset:]
    guard = wl.bf16_bits(torch.tensor([-7.0], dtype=torch.bfloat16))[0]
    want = np.full((T, 576), guard, np.uint16)
    ofn = oracle_mod.gather_nvfp4_ds_mla if entry == 352 else oracle_mod.gather_fp8_ds_mla
    B = len(starts) if batch_size is None else batch_size
    ofn(cache_host, table, np.asarray(ws)[:B], np.asarray(starts)[:B], T, dst=want, threads=threads)
    got = wl.bf16_bits(dst)
    assert int(status.item()) == status_expected
    np.testing.assert_array_equal(got[:, :576], want)
    if dst_pad:
        assert np.all(got[:, 576:] == guard)


def oracle_cache(oracle_mod, w, threads=1):
    c = np.zeros((w.num_blocks, w.block_size, w.entry_bytes), np.uint8)
    fn = oracle_mod.write_nvfp4_ds_mla if w.entry_bytes == 352 else oracle_mod.write_fp8_ds_mla
    fn(wl.bf16_bits(w.kv_c), wl.bf16_bits(w.k_pe), wl.host(w.slot_mapping), c, threads=threads)
    return c


def random_nvfp4_cache(nb, bs, seed):
    c = wl.random_bytes((nb, bs, 352), seed)
    wl.nan_free_e4m3_bytes(c[..., 256:352])
    return c


def random_fp8_cache(nb, bs, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    c = wl.random_bytes((nb, bs, 656), seed + 1)
    wl.nan_free_e4m3_bytes(c[..., :512])
    s = (np.exp2(g.integers(-20, 12, size=(nb, bs, 4))) *
         np.where(g.random((nb, bs, 4)) < 0.5, 1.0, 1.0 + g.random((nb, bs, 4)))).astype("<f4")
    c[..., 512:528] = s.view(np.uint8).reshape(nb, bs, 16)
    return c


GATHER_CASES = [
    # name, (nb, bs), lens, starts, extra
    ("two requests", (8, 64), [100, 120], [0, 17], {}),
    ("zero-length and block-edge starts", (16, 64), [0, 64, 1, 0, 130], [0, 64, 63, 5, 0], {}),
    ("ragged rows T=130", (8, 64), [130], [1], {}),
    ("block_size 16, padded strides", (64, 16), [77, 5, 200], [15, 16, 31],
     dict(pad_entry=32, pad_block=1, dst_pad=64)),
    ("300 short requests", (4096, 16), list(range(1, 301)), [i % 40 for i in range(300)], {}),
    ("block_size 7", (200, 7), [90, 0, 300, 17], [6, 3, 0, 13], {}),
    ("block_size 48", (40, 48), [500, 333], [47, 1], {}),
    ("16-byte aligned rows", (16, 64), [130, 70], [5, 64], dict(dst_offset=8, dst_pad=16)),
]


@pytest.mark.parametrize("entry", [352, 656])
@pytest.mark.parametrize("name,geom,lens,starts,kw", GATHER_CASES, ids=[c[0] for c in GATHER_CASES])
def test_gather_parity_random_cache(kvq, oracle_mod, entry, name, geom, lens, starts, kw):
    nb, bs = geom
    cache = random_nvfp4_cache(nb, bs, 81) if entry == 352 else random_fp8_cache(nb, bs, 82)
    table, ws, st, T = wl.make_gather_batch(nb, bs, lens, starts, 83)
    run_gather(kvq, oracle_mod, entry, cache, table, ws, st, T, **kw)


@pytest.mark.parametrize("entry", [352, 656])
def test_gather_of_written_cache(kvq, oracle_mod, entry):
    fill = wl.make_fill("f", 8, 64, 84, entry_bytes=entry)
    cache = oracle_cache(oracle_mod, fill)
    table, ws, st, T = wl.make_gather_batch(8, 64, [100, 120], [0, 17], 85)
    run_gather(kvq, oracle_mod, entry, cache, table, ws, st, T)


@pytest.mark.parametrize("entry", [352, 656])
def test_gather_accepts_cu_seq_lens(kvq, oracle_mod, entry):
    cache = random_nvfp4_cache(8, 64, 86) if entry == 352 else random_fp8_cache(8, 64, 86)
    table, ws, st, T = wl.make_gather_batch(8, 64, [50, 70, 30], [3, 0, 9], 87)
    cu = np.concatenate([ws, [T]]).astype(np.int32)
    run_gather(kvq, oracle_mod, entry, cache, table, cu, st, T, batch_size=3)


@pytest.mark.parametrize("entry", [352, 656])
def test_gather_bad_block_ids_skip_rows_and_report(kvq, oracle_mod, entry):
    cache = random_nvfp4_cache(8, 64, 88) if entry == 352 else random_fp8_cache(8, 64, 88)
    table, ws, st, T = wl.make_gather_batch(8, 64, [100, 120], [0, 17], 89)
    table = table.copy()
    table[0, 1] = 8            # one past the last block
    table[1, 0] = -1
    run_gather(kvq, oracle_mod, entry, cache, table, ws, st, T, status_expected=kvq.STATUS_BAD_INDEX)


def test_gather_non_monotone_workspace_starts_reported(kvq):
    cache = dev(random_nvfp4_cache(8, 64, 90))
    table, _, st, _ = wl.make_gather_batch(8, 64, [50, 50], [0, 0], 91)
    dst = torch.zeros((100, 576), dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvq.kvq_gather_upconvert_nvfp4_ds_mla(cache, dst, dev(table), dev(np.array([60, 10], np.int32)),
                                          dev(st), status=status)
    assert int(status.item()) & kvq.STATUS_BAD_BATCH


def test_gather_prefill_full_size(kvq, oracle_mod, threads):
    """32 requests of 4k-32k rows over the 65536 x 64 cache written by the
    GPU fill: cache and every gathered row against the oracle."""
    g = wl.prefill_gather(DEV)
    w = g.fill
    cache = torch.zeros((w.num_blocks, w.block_size, 352), dtype=torch.uint8, device=DEV)
    kvq.kvq_write_nvfp4_ds_mla(w.kv_c, w.k_pe, cache, w.slot_mapping)
    dst = torch.empty((g.num_out_tokens, 576), dtype=torch.bfloat16, device=DEV)
    kvq.kvq_gather_upconvert_nvfp4_ds_mla(cache, dst, g.block_table, g.workspace_starts, g.seq_starts)
    ocache = oracle_cache(oracle_mod, w, threads)
    got_cache = cache.cpu().numpy()
    assert np.array_equal(got_cache, ocache)
    del got_cache
    want, skipped = oracle_mod.gather_nvfp4_ds_mla(ocache, wl.host(g.block_table), wl.host(g.workspace_starts),
                                                   wl.host(g.seq_starts), g.num_out_tokens, threads=threads)
    assert skipped == 0
    got = wl.bf16_bits(dst)
    assert np.array_equal(got, want), f"{int((got != want).sum())} values differ"


def test_gather_fp8_full_size(kvq, oracle_mod, threads):
    """16 requests x 16384 rows over the 32768 x 64 x 656 cache written by the
    GPU fp8 fill: cache and every gathered row against the oracle."""
    g = wl.fp8_gather(DEV)
    w = g.fill
    cache = torch.zeros((w.num_blocks, w.block_size, 656), dtype=torch.uint8, device=DEV)
    kvq.kvq_write_fp8_ds_mla(w.kv_c, w.k_pe, cache, w.slot_mapping)
    dst = torch.empty((g.num_out_tokens, 576), dtype=torch.bfloat16, device=DEV)
    kvq.kvq_gather_upconvert_fp8_ds_mla(cache, dst, g.block_table, g.workspace_starts, g.seq_starts)
    ocache = oracle_cache(oracle_mod, w, threads)
    got_cache = cache.cpu().numpy()
    assert np.array_equal(got_cache, ocache)
    del got_cache
    want, skipped = oracle_mod.gather_fp8_ds_mla(ocache, wl.host(g.block_table), wl.host(g.workspace_starts),
                                                 wl.host(g.seq_starts), g.num_out_tokens, threads=threads)
    assert skipped == 0
    got = wl.bf16_bits(dst)
    assert np.array_equal(got, want), f"{int((got != want).sum())} values differ"


# --------------------------------------------------------------------------
# per-head NVFP4 cache
# --------------------------------------------------------------------------

def per_head_shape(w, kvq, layout):
    T, H, D = w.key.shape
    fd = kvq.nvfp4_full_dim(D)
    if layout == "HND":
        return (w.num_pages, 2, H, w.block_size, fd)
    return (w.num_pages, 2, w.block_size, H, fd)


def run_per_head(kvq, oracle_mod, w, strided=False, status_expected=0, threads=1, narrow_rows=False,
                 layout="NHD"):
    T, H, D = w.key.shape
    init = wl.random_bytes(per_head_shape(w, kvq, layout), 5)
    cache = dev(init.copy())
    if strided:            # key and value as interleaved halves of one [T, H, 2D] tensor
        both = torch.cat([w.key, w.value], dim=2).to(DEV)
        key, value = both[:, :, :D], both[:, :, D:]
    elif narrow_rows:      # 16-byte but not 32-byte aligned groups: the two-access path
        kb = torch.zeros((T, H, D + 24), dtype=torch.bfloat16, device=DEV)
        vb = torch.zeros((T, H, D + 24), dtype=torch.bfloat16, device=DEV)
        kb[:, :, 8:8 + D] = w.key.to(DEV)
        vb[:, :, 8:8 + D] = w.value.to(DEV)
        key, value = kb[:, :, 8:8 + D], vb[:, :, 8:8 + D]
    else:
        key, value = dev(w.key), dev(w.value)
    ks = torch.tensor([w.k_scale], dtype=torch.float32, device=DEV)
    vs = torch.tensor([w.v_scale], dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvq.kvq_reshape_and_cache_nvfp4(key, value, cache, dev(w.slot_mapping), ks, vs, status=status,
                                    layout=layout)
    want = init.copy()
    oracle_mod.reshape_and_cache_nvfp4(wl.bf16_bits(w.key), wl.bf16_bits(w.value), wl.host(w.slot_mapping),
                                       want, w.k_scale, w.v_scale, threads=threads, layout=layout)
    assert int(status.item()) == status_expected
    got = cache.cpu().numpy()
    assert np.array_equal(got, want), f"{int((got != want).sum())} bytes differ"


PER_HEAD_CASES = [
    ("H8 D128", lambda: wl.make_per_head("a", 333, 8, 128, 64, 16, 11, 101), {}),
    ("H1 D64 scales", lambda: wl.make_per_head("b", 100, 1, 64, 16, 16, 3, 102, k_scale=0.75,
                                               v_scale=3.0), {}),
    ("H4 D256", lambda: wl.make_per_head("c", 77, 4, 256, 8, 16, 0, 103, k_scale=2.0), {}),
    ("H8 D128 strided", lambda: wl.make_per_head("d", 129, 8, 128, 32, 16, 4, 104), dict(strided=True)),
    ("block_size 1", lambda: wl.make_per_head("e", 50, 8, 128, 64, 1, 2, 105), {}),
    ("H3 D48 block_size 24", lambda: wl.make_per_head("f", 90, 3, 48, 12, 24, 4, 107, v_scale=1.5), {}),
    ("16-byte aligned rows", lambda: wl.make_per_head("g", 45, 4, 128, 8, 16, 2, 108), dict(narrow_rows=True)),
    ("H1 D32 block_size 4 (8-byte aligned regions)", lambda: wl.make_per_head("h", 50, 1, 32, 40, 4, 2, 109), {}),
]


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("name,make,kw", PER_HEAD_CASES, ids=[c[0] for c in PER_HEAD_CASES])
def test_per_head_parity(kvq, oracle_mod, name, make, kw, layout):
    run_per_head(kvq, oracle_mod, make(), layout=layout, **kw)


@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.75, 3.0), (2.0 ** -20, 2.0 ** 20)])
def test_per_head_parity_extreme_values(kvq, oracle_mod, k_scale, v_scale):
    """Random finite bf16 bit patterns (subnormals, zeros, values up to the bf16
    maximum, so x / scale can overflow to infinity) and zero groups."""
    T, H, D = 64, 4, 64
    kb = finite_bf16_bits((T, H, D), 151)
    vb = finite_bf16_bits((T, H, D), 152)
    kb[3] = 0
    vb[4] = 0x8000
    slots = wl.slot_mapping(T, 16 * 8, 5, 153)
    w = wl.PerHeadWorkload("extreme", bits_to_bf16(kb), bits_to_bf16(vb), torch.from_numpy(slots), 8, 16,
                           k_scale, v_scale)
    run_per_head(kvq, oracle_mod, w)


def test_per_head_out_of_range_slots(kvq, oracle_mod):
    w = wl.make_per_head("oob", 40, 8, 128, 4, 16, 2, 106)
    s = wl.host(w.slot_mapping).copy()
    s[[0, 7]] = [64, 1000]
    w.slot_mapping = torch.from_numpy(s)
    run_per_head(kvq, oracle_mod, w, status_expected=kvq.STATUS_BAD_INDEX)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_per_head_full_size(kvq, oracle_mod, threads, layout):
    run_per_head(kvq, oracle_mod, wl.per_head(), threads=threads, layout=layout)


# --------------------------------------------------------------------------
# per-head read-back (next row: the consumer side of the per-head cache)
# --------------------------------------------------------------------------

def run_dequant(kvq, oracle_mod, w, cache_host, strided=False, status_expected=0, threads=1,
                narrow_rows=False, layout="NHD"):
    T, H, D = w.key.shape
    if strided:          # outputs as halves of one [T, H, 2D] tensor
        both = torch.full((T, H, 2 * D), -3.0, dtype=torch.bfloat16, device=DEV)
        ko, vo = both[:, :, :D], both[:, :, D:]
    elif narrow_rows:    # 16-byte but not 32-byte aligned output groups
        kb = torch.full((T, H, D + 24), -3.0, dtype=torch.bfloat16, device=DEV)
        vb = torch.full((T, H, D + 24), -3.0, dtype=torch.bfloat16, device=DEV)
        ko, vo = kb[:, :, 8:8 + D], vb[:, :, 8:8 + D]
    else:
        ko = torch.full((T, H, D), -3.0, dtype=torch.bfloat16, device=DEV)
        vo = torch.full((T, H, D), -3.0, dtype=torch.bfloat16, device=DEV)
    ks = torch.tensor([w.k_scale], dtype=torch.float32, device=DEV)
    vs = torch.tensor([w.v_scale], dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvq.kvq_dequant_nvfp4_per_head(dev(cache_host), dev(w.slot_mapping), ks, vs, ko, vo, status=status,
                                   layout=layout)
    guard = wl.bf16_bits(torch.tensor([-3.0], dtype=torch.bfloat16))[0]
    wk = np.full((T, H, D), guard, np.uint16)
    wv = np.full((T, H, D), guard, np.uint16)
    oracle_mod.dequant_nvfp4_per_head(cache_host, wl.host(w.slot_mapping), H, D, w.k_scale, w.v_scale,
                                      key_out=wk, value_out=wv, threads=threads, layout=layout)
    assert int(status.item()) == status_expected
    np.testing.assert_array_equal(wl.bf16_bits(ko), wk)
    np.testing.assert_array_equal(wl.bf16_bits(vo), wv)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("name,make,kw", PER_HEAD_CASES, ids=[c[0] for c in PER_HEAD_CASES])
def test_dequant_per_head_parity_written_cache(kvq, oracle_mod, name, make, kw, layout):
    w = make()
    cache = np.zeros(per_head_shape(w, kvq, layout), np.uint8)
    oracle_mod.reshape_and_cache_nvfp4(wl.bf16_bits(w.key), wl.bf16_bits(w.value), wl.host(w.slot_mapping),
                                       cache, w.k_scale, w.v_scale, layout=layout)
    run_dequant(kvq, oracle_mod, w, cache, layout=layout, **kw)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_dequant_per_head_random_cache_and_bad_slots(kvq, oracle_mod, layout):
    w = wl.make_per_head("rb", 70, 4, 64, 8, 16, 5, 111, k_scale=0.3, v_scale=7.0)
    s = wl.host(w.slot_mapping).copy()
    s[[1, 2]] = [128, 999]
    w.slot_mapping = torch.from_numpy(s)
    cache = wl.random_bytes(per_head_shape(w, kvq, layout), 112)
    # scale bytes must be finite e4m3: every byte that can be a scale byte
    wl.nan_free_e4m3_bytes(cache)
    run_dequant(kvq, oracle_mod, w, cache, status_expected=kvq.STATUS_BAD_INDEX, layout=layout)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_dequant_per_head_full_size(kvq, oracle_mod, threads, layout):
    w = wl.per_head()
    T, H, D = w.key.shape
    shape = (w.block_size, H) if layout == "NHD" else (H, w.block_size)
    cache = np.zeros((w.num_pages, 2, *shape, kvq.nvfp4_full_dim(D)), np.uint8)
    oracle_mod.reshape_and_cache_nvfp4(wl.bf16_bits(w.key), wl.bf16_bits(w.value), wl.host(w.slot_mapping),
                                       cache, threads=threads, layout=layout)
    run_dequant(kvq, oracle_mod, w, cache, threads=threads, layout=layout)


# --------------------------------------------------------------------------
# sparse-decode index conversion (next row)
# --------------------------------------------------------------------------

def index_case(num_req, lens, bs, nb, N, topk, seed, p_unused=0.2):
    g = np.random.Generator(np.random.PCG64(seed))
    table, _, _, _ = wl.make_gather_batch(nb, bs, lens, [0] * len(lens), seed)
    req = g.integers(0, num_req, size=N).astype(np.int32)
    lens = np.asarray(lens)
    idx = (g.random((N, topk)) * lens[req][:, None]).astype(np.int32)
    idx[g.random((N, topk)) < p_unused] = -1
    return req, idx, table


@pytest.mark.parametrize("bs,topk", [(64, 2048), (16, 100), (7, 33), (1, 8)])
def test_index_conversion_parity(kvq, oracle_mod, bs, topk):
    req, idx, table = index_case(6, [5000, 1, 300, 2048, 64, 999], bs, 20000, 77, topk, 121 + bs)
    out = kvq.kvq_req_index_to_global_slot(dev(req), dev(idx), dev(table), bs, 20000)
    want, skipped = oracle_mod.req_index_to_global_slot(req, idx, table, bs, 20000)
    assert skipped == 0
    np.testing.assert_array_equal(out.cpu().numpy(), want)


def test_index_conversion_strided_rows_and_bad_entries(kvq, oracle_mod):
    req, idx, table = index_case(3, [100, 200, 50], 16, 64, 40, 24, 131)
    req[5] = 7                      # no such request
    idx[6, 3] = 10 ** 6             # past the block table
    table = table.copy()
    table[1, 0] = -1                # unusable block
    wide = np.full((40, 32), 5, np.int32)
    wide[:, :24] = idx
    ti = dev(wide)[:, :24]
    outbuf = torch.full((40, 30), 99, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvq.kvq_req_index_to_global_slot(dev(req), ti, dev(table), 16, 64, out=outbuf[:, :24], status=status)
    want, skipped = oracle_mod.req_index_to_global_slot(req, idx, table, 16, 64)
    assert skipped > 0 and int(status.item()) == kvq.STATUS_BAD_INDEX
    got = outbuf.cpu().numpy()
    np.testing.assert_array_equal(got[:, :24], want)
    assert np.all(got[:, 24:] == 99)


def test_index_conversion_rejects_length_mismatch(kvq):
    req, idx, table = index_case(2, [10, 10], 16, 8, 12, 4, 141)
    with pytest.raises(RuntimeError, match="req_id has 13 entries"):
        kvq.kvq_req_index_to_global_slot(dev(np.concatenate([req, [0]]).astype(np.int32)), dev(idx),
                                         dev(table), 16, 8)


# --------------------------------------------------------------------------
# stream capture: the entry points allocate nothing and never synchronise,
# so a sequence of them can be captured in a CUDA graph and replayed
# --------------------------------------------------------------------------

def test_entry_points_replay_from_a_cuda_graph(kvq):
    g = wl.smoke_gather(DEV)
    f = g.fill
    ph = wl.make_per_head("graph", 64, 8, 128, 16, 16, 3, 161, DEV, k_scale=0.5)
    ks = torch.tensor([ph.k_scale], device=DEV)
    vs = torch.tensor([ph.v_scale], device=DEV)

    def run(c352, c656, ws352, ws656, phc, ko, vo):
        kvq.kvq_write_nvfp4_ds_mla(f.kv_c, f.k_pe, c352, f.slot_mapping)
        kvq.kvq_write_fp8_ds_mla(f.kv_c, f.k_pe, c656, f.slot_mapping)
        kvq.kvq_gather_upconvert_nvfp4_ds_mla(c352, ws352, g.block_table, g.workspace_starts, g.seq_starts)
        kvq.kvq_gather_upconvert_fp8_ds_mla(c656, ws656, g.block_table, g.workspace_starts, g.seq_starts)
        kvq.kvq_reshape_and_cache_nvfp4(ph.key, ph.value, phc, ph.slot_mapping, ks, vs)
        kvq.kvq_dequant_nvfp4_per_head(phc, ph.slot_mapping, ks, vs, ko, vo)

    def buffers():
        return (torch.zeros((8, 64, 352), dtype=torch.uint8, device=DEV),
                torch.zeros((8, 64, 656), dtype=torch.uint8, device=DEV),
                torch.zeros((g.num_out_tokens, 576), dtype=torch.bfloat16, device=DEV),
                torch.zeros((g.num_out_tokens, 576), dtype=torch.bfloat16, device=DEV),
                torch.zeros((16, 2, 16, 8, 72), dtype=torch.uint8, device=DEV),
                torch.zeros_like(ph.key), torch.zeros_like(ph.value))

    direct = buffers()
    run(*direct)
    captured = buffers()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run(*captured)                      # warm-up outside capture
    torch.cuda.current_stream().wait_stream(side)
    for t in captured:
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(*captured)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(direct, captured):
        assert torch.equal(a.view(torch.uint8) if a.dtype == torch.uint8 else a.view(torch.int16),
                           b.view(torch.uint8) if b.dtype == torch.uint8 else b.view(torch.int16))


# --------------------------------------------------------------------------
# gather index walk: more than 1024 requests (starts searched in global
# memory instead of shared memory), rows before the first request
# --------------------------------------------------------------------------

@pytest.mark.parametrize("entry", [352, 656])
def test_gather_more_requests_than_staged_in_shared_memory(kvq, oracle_mod, entry):
    g = np.random.Generator(np.random.PCG64(181))
    B = 1500
    lens = g.integers(0, 9, size=B)
    starts = g.integers(0, 40, size=B)
    nb, bs = 3200, 16
    cache = random_nvfp4_cache(nb, bs, 182) if entry == 352 else random_fp8_cache(nb, bs, 182)
    table, ws, st, T = wl.make_gather_batch(nb, bs, lens, starts, 183)
    run_gather(kvq, oracle_mod, entry, cache, table, ws, st, T)


@pytest.mark.parametrize("entry", [352, 656])
def test_gather_rows_before_the_first_request_are_skipped(kvq, oracle_mod, entry):
    cache = random_nvfp4_cache(8, 64, 191) if entry == 352 else random_fp8_cache(8, 64, 191)
    table, ws, st, T = wl.make_gather_batch(8, 64, [40, 30], [3, 9], 192)
    ws = ws + 5                      # rows 0..4 belong to no request
    run_gather(kvq, oracle_mod, entry, cache, table, ws, st, T + 5, status_expected=kvq.STATUS_BAD_BATCH)
