"""Pins of the oracle's operations (CPU only).

Each op is checked against an independent restatement built from torch's
float8/bf16 casts and the exhaustive encoders in tests/independent.py, and
against closed forms and invariants the pages fix: entry sizes and region
offsets, the padding rule, the slot -> (block, offset) decomposition, exact
round trips for values on the format's grid, and the error bounds of the
NVFP4 DS-MLA page's test (scale bytes within 1 e4m3 ulp, NoPE error
<= 1.5 sf, RoPE error <= |x| 2^-3 + 2^-9).
"""
import numpy as np
import pytest
import torch

import independent as ind
import workloads as wl

E4M3 = ind.e4m3_table()
E2M1 = ind.e2m1_table()


# --------------------------------------------------------------------------
# independent restatements (numpy + torch casts)
# --------------------------------------------------------------------------

def ref_nvfp4_groups(x: np.ndarray):
    """x float32 [..., 16k] -> (packed uint8 [..., 8k], sf uint8 [..., k])."""
    shape = x.shape
    g = x.reshape(*shape[:-1], shape[-1] // 16, 16)
    amax = np.abs(g).max(axis=-1).astype(np.float32)
    sf = ind.torch_e4m3_bits(torch.from_numpy((amax / np.float32(6.0)).astype(np.float32))).numpy()
    sfv = E4M3[sf].astype(np.float32)
    inv = np.zeros_like(sfv)
    np.divide(np.float32(1.0), sfv, out=inv, where=sfv != 0)
    y = (g * inv[..., None]).astype(np.float32)
    codes = ind.e2m1_encode(y).reshape(g.shape)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    return packed.reshape(*shape[:-1], shape[-1] // 2), sf


def ref_nvfp4_entries(kv_c_bits: np.ndarray, k_pe_bits: np.ndarray) -> np.ndarray:
    x = ind.bf16_to_f32(kv_c_bits)
    packed, sf = ref_nvfp4_groups(x)
    rope = ind.torch_e4m3_bits(torch.from_numpy(ind.bf16_to_f32(k_pe_bits).copy())).numpy()
    return np.concatenate([packed, rope, sf], axis=1)


def ref_fp8_entries(kv_c_bits: np.ndarray, k_pe_bits: np.ndarray) -> np.ndarray:
    x = ind.bf16_to_f32(kv_c_bits).reshape(-1, 4, 128)
    amax = np.abs(x).max(axis=-1).astype(np.float32)
    s = np.where(amax == 0, np.float32(1.0), amax / np.float32(448.0)).astype(np.float32)
    q = ind.torch_e4m3_bits(torch.from_numpy((x / s[..., None]).astype(np.float32))).numpy()
    return np.concatenate([q.reshape(-1, 512), s.view(np.uint8).reshape(-1, 16),
                           k_pe_bits.astype("<u2").view(np.uint8).reshape(-1, 128)], axis=1)


def host_write(w: wl.WriteWorkload):
    return wl.bf16_bits(w.kv_c), wl.bf16_bits(w.k_pe), wl.host(w.slot_mapping)


def random_cache(w: wl.WriteWorkload, seed=77):
    return wl.random_bytes((w.num_blocks, w.block_size, w.entry_bytes), seed)


# --------------------------------------------------------------------------
# format constants
# --------------------------------------------------------------------------

def test_layout_constants_match_pages(oracle_mod):
    g = {k: int(v) for k, v in ind.read_golden("entry_layout.txt")}
    assert oracle_mod.nvfp4_ds_mla_entry_bytes() == g["nvfp4_ds_mla_entry"]
    assert g["nvfp4_nope_bytes"] + g["nvfp4_rope_bytes"] + g["nvfp4_sf_bytes"] == g["nvfp4_ds_mla_entry"]
    assert oracle_mod.fp8_ds_mla_entry_bytes() == g["fp8_ds_mla_entry"]
    for d in (64, 128, 256):
        fd = oracle_mod.nvfp4_full_dim(d)
        assert fd == g[f"full_dim_{d}"]
        assert oracle_mod.nvfp4_data_dim(fd) == g[f"data_dim_{fd}"] == d // 2
        assert oracle_mod.nvfp4_scale_dim(fd) == g[f"scale_dim_{fd}"] == d // 16
    # per-head page bytes at 16 tokens x 8 heads x head_size 128
    assert 2 * 16 * 8 * oracle_mod.nvfp4_full_dim(128) == 18432


# --------------------------------------------------------------------------
# nvfp4_ds_mla write
# --------------------------------------------------------------------------

def test_write_matches_independent_restatement(oracle_mod):
    w = wl.smoke_write()
    kv, pe, slots = host_write(w)
    cache0 = random_cache(w)
    cache = cache0.copy()
    assert oracle_mod.write_nvfp4_ds_mla(kv, pe, slots, cache) == 0
    want = cache0.copy().reshape(-1, 352)
    valid = slots >= 0
    want[slots[valid]] = ref_nvfp4_entries(kv[valid], pe[valid])
    np.testing.assert_array_equal(cache.reshape(-1, 352), want)


def test_write_decode_step_with_outliers_matches_restatement(oracle_mod):
    w = wl.decode_write()
    kv, pe, slots = host_write(w)
    cache = np.zeros((w.num_blocks, w.block_size, 352), np.uint8)
    oracle_mod.write_nvfp4_ds_mla(kv, pe, slots, cache, threads=4)
    valid = slots >= 0
    np.testing.assert_array_equal(cache.reshape(-1, 352)[slots[valid]],
                                  ref_nvfp4_entries(kv[valid], pe[valid]))


def test_write_closed_form_grid_values_round_trip(oracle_mod):
    """x = c * S with e2m1 codes c (max |c| = 6 per group) and an e4m3 normal
    S encodes to exactly c and sf = S; e4m3-representable RoPE is exact."""
    g = np.random.Generator(np.random.PCG64(11))
    T = 64
    sf_codes = g.integers(0x20, 0x61, size=(T, 32)).astype(np.uint8)   # 2^-3 .. 2^5
    codes = g.integers(0, 16, size=(T, 32, 16)).astype(np.uint8)
    codes[np.arange(T)[:, None], np.arange(32)[None, :], g.integers(0, 16, size=(T, 32))] = \
        g.choice([0x7, 0xF], size=(T, 32))
    x = E2M1[codes] * E4M3[sf_codes][..., None]
    kv = ind.torch_bf16_bits(torch.from_numpy(x.reshape(T, 512).astype(np.float32)))
    assert np.array_equal(ind.bf16_to_f32(kv).astype(np.float64), x.reshape(T, 512))  # exact
    rope_codes = g.integers(0, 256, size=(T, 64)).astype(np.uint8)
    rope_codes[(rope_codes & 0x7F) == 0x7F] = 0x38
    pe = ind.torch_bf16_bits(torch.from_numpy(E4M3[rope_codes].astype(np.float32)))
    slots = np.arange(T, dtype=np.int64)
    cache = np.zeros((1, T, 352), np.uint8)
    oracle_mod.write_nvfp4_ds_mla(kv, pe, slots, cache)
    e = cache[0]
    np.testing.assert_array_equal(e[:, 320:], sf_codes)
    np.testing.assert_array_equal(ind.unpack_e2m1(e[:, :256]).reshape(T, 32, 16), codes)
    # rope: -0 and +0 are distinct codes and must survive
    np.testing.assert_array_equal(e[:, 256:320], rope_codes)


def test_write_padding_and_untouched_bytes(oracle_mod):
    w = wl.smoke_write()
    kv, pe, slots = host_write(w)
    slots = slots.copy()
    slots[[0, 1, 2]] = [-7, np.iinfo(np.int64).min, -2]       # any negative slot is padding
    cache0 = random_cache(w, 5)
    cache = cache0.copy()
    assert oracle_mod.write_nvfp4_ds_mla(kv, pe, slots, cache) == 0
    written = np.zeros(w.num_slots, bool)
    written[slots[slots >= 0]] = True
    flat0, flat = cache0.reshape(-1, 352), cache.reshape(-1, 352)
    np.testing.assert_array_equal(flat[~written], flat0[~written])
    assert np.any(flat[written] != flat0[written])


def test_write_out_of_range_slot_is_skipped_and_counted(oracle_mod):
    w = wl.smoke_write()
    kv, pe, slots = host_write(w)
    slots = slots.copy()
    slots[5] = w.num_slots          # one past the end
    slots[6] = w.num_slots * 10
    cache0 = random_cache(w, 6)
    cache = cache0.copy()
    assert oracle_mod.write_nvfp4_ds_mla(kv, pe, slots, cache) == 2


def test_write_slot_decomposition_and_strides(oracle_mod):
    """A cache with padded entries and padded blocks: slot s lands at
    (s // block_size) * block_stride + (s % block_size) * entry_stride."""
    w = wl.make_write("strided", 50, 3, 32, 4, 99)
    kv, pe, slots = host_write(w)
    big = np.zeros((3, 33, 368), np.uint8)                       # block 33*368 B, entry 368 B
    view = big[:, :32, :352]
    oracle_mod.write_nvfp4_ds_mla(kv, pe, slots, view)
    ref = ref_nvfp4_entries(kv, pe)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        np.testing.assert_array_equal(big[s // 32, s % 32, :352], ref[t])
    assert not big[:, 32].any() and not big[:, :, 352:].any()


def test_write_region_of_each_input_element(oracle_mod):
    """Changing NoPE element k moves only its group's 8 data bytes and its
    scale byte; changing RoPE element j moves only byte 256 + j."""
    w = wl.make_write("one", 1, 1, 1, 0, 123)
    kv, pe, slots = host_write(w)
    base = np.zeros((1, 1, 352), np.uint8)
    oracle_mod.write_nvfp4_ds_mla(kv, pe, slots, base)
    for k in (0, 1, 17, 255, 256, 511):
        kv2 = kv.copy()
        kv2[0, k] = ind.torch_bf16_bits(torch.tensor([37.0]))[0]
        c = np.zeros_like(base)
        oracle_mod.write_nvfp4_ds_mla(kv2, pe, slots, c)
        changed = set(np.nonzero(c[0, 0] != base[0, 0])[0].tolist())
        gidx = k // 16
        assert k // 2 in changed
        assert changed <= set(range(8 * gidx, 8 * gidx + 8)) | {320 + gidx}
    for j in (0, 9, 63):
        pe2 = pe.copy()
        pe2[0, j] = ind.torch_bf16_bits(torch.tensor([-3.0]))[0]
        c = np.zeros_like(base)
        oracle_mod.write_nvfp4_ds_mla(kv, pe2, slots, c)
        assert set(np.nonzero(c[0, 0] != base[0, 0])[0].tolist()) == {256 + j}


def test_write_error_bounds_of_the_reference_test(oracle_mod):
    """NVFP4 DS-MLA page, test_cache.py: sf within 1 e4m3 ulp of
    e4m3(amax / 6), NoPE error <= 1.5 sf, RoPE error <= |x| 2^-3 + 2^-9."""
    w = wl.decode_write()
    kv, pe, slots = host_write(w)
    cache = np.zeros((w.num_blocks, w.block_size, 352), np.uint8)
    oracle_mod.write_nvfp4_ds_mla(kv, pe, slots, cache, threads=4)
    valid = np.nonzero(slots >= 0)[0][:2000]
    e = cache.reshape(-1, 352)[slots[valid]]
    x = ind.bf16_to_f32(kv[valid]).astype(np.float64)
    r = ind.bf16_to_f32(pe[valid]).astype(np.float64)
    amax = np.abs(x.reshape(-1, 32, 16)).max(-1).astype(np.float32)
    ref_sf = ind.torch_e4m3_bits(torch.from_numpy(amax / np.float32(6))).numpy()
    assert np.abs(e[:, 320:].astype(int) - ref_sf.astype(int)).max() <= 1
    sf = np.repeat(E4M3[e[:, 320:]], 16, axis=1)
    nope = E2M1[ind.unpack_e2m1(e[:, :256])] * sf
    assert np.all(np.abs(nope - x) <= 1.5 * sf)
    rope = E4M3[e[:, 256:320]]
    assert np.all(np.abs(rope - r) <= np.abs(r) * 2.0 ** -3 + 2.0 ** -9)


def test_write_zero_group_gives_zero_scale_and_signed_zero_codes(oracle_mod):
    kv = np.zeros((1, 512), np.uint16)
    kv[0, 16:32] = 0x8000                                    # -0.0 in group 1
    kv[0, 32] = 0x0001                                       # tiny subnormal in group 2
    pe = np.zeros((1, 64), np.uint16)
    cache = np.full((1, 1, 352), 0xAA, np.uint8)
    oracle_mod.write_nvfp4_ds_mla(kv, pe, np.zeros(1, np.int64), cache)
    e = cache[0, 0]
    assert e[320] == 0 and e[321] == 0 and e[322] == 0
    assert np.all(e[0:8] == 0) and np.all(e[8:16] == 0x88)
    assert np.all(e[256:320] == 0)


# --------------------------------------------------------------------------
# nvfp4_ds_mla gather
# --------------------------------------------------------------------------

def brute_gather_rows(cache_flat, bs, table, ws, starts, T, entry_fn):
    """Row-by-row restatement of the gather's index walk."""
    rows = []
    for w in range(T):
        b = max(i for i in range(len(ws)) if ws[i] <= w)
        p = starts[b] + (w - ws[b])
        blk = table[b][p // bs]
        rows.append(entry_fn(cache_flat[blk * bs + p % bs]))
    return np.stack(rows)


def nvfp4_entry_bf16(e):
    vals = np.concatenate([E2M1[ind.unpack_e2m1(e[:256])] * np.repeat(E4M3[e[320:352]], 16),
                           E4M3[e[256:320]]])
    return ind.torch_bf16_bits(torch.from_numpy(vals.astype(np.float32)))


def fp8_entry_bf16(e):
    s = e[512:528].view("<f4").astype(np.float32)
    vals = (E4M3[e[:512]].astype(np.float32).reshape(4, 128) * s[:, None]).astype(np.float32)
    return np.concatenate([ind.torch_bf16_bits(torch.from_numpy(vals.reshape(512))),
                           e[528:656].view("<u2")])


def oracle_filled(oracle_mod, g: wl.GatherWorkload):
    kv, pe, slots = host_write(g.fill)
    cache = np.zeros((g.fill.num_blocks, g.fill.block_size, g.fill.entry_bytes), np.uint8)
    fn = oracle_mod.write_nvfp4_ds_mla if g.fill.entry_bytes == 352 else oracle_mod.write_fp8_ds_mla
    fn(kv, pe, slots, cache, threads=4)
    return cache


def test_gather_matches_bruteforce_walk(oracle_mod):
    g = wl.smoke_gather()
    cache = oracle_filled(oracle_mod, g)
    table, ws, st = wl.host(g.block_table), wl.host(g.workspace_starts), wl.host(g.seq_starts)
    out, skipped = oracle_mod.gather_nvfp4_ds_mla(cache, table, ws, st, g.num_out_tokens)
    assert skipped == 0 and out.shape == (220, 576)
    want = brute_gather_rows(cache.reshape(-1, 352), 64, table, ws, st, 220, nvfp4_entry_bf16)
    np.testing.assert_array_equal(out, want)


def test_gather_of_write_is_quantize_dequantize(oracle_mod):
    """Row w holds the qdq of the token written to its slot: equal to the
    decoded entry, and within the reference test's bounds of the input."""
    g = wl.smoke_gather()
    kv, pe, slots = host_write(g.fill)
    cache = oracle_filled(oracle_mod, g)
    table, ws, st = wl.host(g.block_table), wl.host(g.workspace_starts), wl.host(g.seq_starts)
    out, _ = oracle_mod.gather_nvfp4_ds_mla(cache, table, ws, st, g.num_out_tokens)
    token_of_slot = np.empty(g.fill.num_slots, np.int64)
    token_of_slot[slots] = np.arange(slots.size)
    for w_ in (0, 57, 99, 100, 150, 219):
        b = 0 if w_ < 100 else 1
        p = st[b] + w_ - ws[b]
        t = token_of_slot[table[b][p // 64] * 64 + p % 64]
        x = ind.bf16_to_f32(kv[t]).astype(np.float64)
        got = ind.bf16_to_f32(out[w_]).astype(np.float64)
        dec = oracle_mod.decode_nvfp4_ds_mla_entry(cache.reshape(-1, 352)[table[b][p // 64] * 64 + p % 64])
        np.testing.assert_array_equal(got, dec)
        sf = np.repeat(E4M3[cache.reshape(-1, 352)[table[b][p // 64] * 64 + p % 64][320:]], 16)
        assert np.all(np.abs(got[:512] - x) <= 1.5 * sf)


def test_gather_single_request_from_zero_is_contiguous_dequant(oracle_mod):
    w = wl.make_fill("f", 4, 16, 21)
    cache = np.zeros((4, 16, 352), np.uint8)
    oracle_mod.write_nvfp4_ds_mla(*host_write(w), cache)
    table = np.array([[2, 0, 3, 1]], np.int32)
    out, skipped = oracle_mod.gather_nvfp4_ds_mla(cache, table, [0], [0], 64)
    assert skipped == 0
    flat = cache[table[0]].reshape(64, 352)
    np.testing.assert_array_equal(out, np.stack([nvfp4_entry_bf16(e) for e in flat]))


def test_gather_zero_length_requests_and_bad_indices(oracle_mod):
    w = wl.make_fill("f", 8, 16, 22)
    cache = np.zeros((8, 16, 352), np.uint8)
    oracle_mod.write_nvfp4_ds_mla(*host_write(w), cache)
    lens, starts = [0, 20, 0, 12], [5, 3, 0, 30]
    table, ws, st, T = wl.make_gather_batch(8, 16, lens, starts, 5)
    assert list(ws) == [0, 0, 20, 20]
    out, skipped = oracle_mod.gather_nvfp4_ds_mla(cache, table, ws, st, T)
    assert skipped == 0
    want = brute_gather_rows(cache.reshape(-1, 352), 16, table, ws, st, T, nvfp4_entry_bf16)
    np.testing.assert_array_equal(out, want)
    # an unusable block id, and a position past the table, are skipped
    bad = table.copy()
    bad[1, 0] = -1
    dst = np.full((T, 576), 0x1234, np.uint16)
    _, skipped = oracle_mod.gather_nvfp4_ds_mla(cache, bad, ws, st, T, dst=dst)
    assert skipped == 13                              # rows 0..12 read block column 0 (positions 3..15)
    assert np.all(dst[:13] == 0x1234) and np.array_equal(dst[13:], want[13:])
    _, skipped = oracle_mod.gather_nvfp4_ds_mla(cache, table, ws, np.array([0, 3, 0, 1000], np.int32), T)
    assert skipped == 12


# --------------------------------------------------------------------------
# fp8_ds_mla write (filler) and gather
# --------------------------------------------------------------------------

def test_fp8_write_matches_independent_restatement(oracle_mod):
    w = wl.make_write("fp8", 300, 8, 64, 12, 31, entry_bytes=656, outlier_p=0.01)
    kv, pe, slots = host_write(w)
    kv = kv.copy()
    kv[3, 128:256] = 0                                 # an all-zero tile: scale 1
    cache0 = random_cache(w)
    cache = cache0.copy()
    oracle_mod.write_fp8_ds_mla(kv, pe, slots, cache)
    want = cache0.reshape(-1, 656).copy()
    v = slots >= 0
    want[slots[v]] = ref_fp8_entries(kv[v], pe[v])
    np.testing.assert_array_equal(cache.reshape(-1, 656), want)
    e3 = cache.reshape(-1, 656)[slots[3]]
    if slots[3] >= 0:
        assert e3[516:520].view("<f4")[0] == 1.0


def test_fp8_gather_matches_bruteforce_and_torch_arithmetic(oracle_mod):
    g = wl.make_gather("fp8g", wl.make_fill("fp8f", 8, 64, 32, entry_bytes=656), [100, 57, 0, 80],
                       [0, 17, 3, 63], 32)
    cache = oracle_filled(oracle_mod, g)
    table, ws, st = wl.host(g.block_table), wl.host(g.workspace_starts), wl.host(g.seq_starts)
    out, skipped = oracle_mod.gather_fp8_ds_mla(cache, table, ws, st, g.num_out_tokens)
    assert skipped == 0
    want = brute_gather_rows(cache.reshape(-1, 656), 64, table, ws, st, g.num_out_tokens, fp8_entry_bf16)
    np.testing.assert_array_equal(out, want)


def test_fp8_gather_power_of_two_scales_are_exact(oracle_mod):
    g = np.random.Generator(np.random.PCG64(33))
    e = wl.nan_free_e4m3_bytes(g.integers(0, 256, size=(1, 16, 656), dtype=np.uint8))
    s = np.exp2(g.integers(-8, 8, size=(16, 4))).astype("<f4")
    e[0, :, 512:528] = s.view(np.uint8).reshape(16, 16)
    table = np.array([[0]], np.int32)
    out, _ = oracle_mod.gather_fp8_ds_mla(e, table, [0], [0], 16)
    vals = ind.bf16_to_f32(out[:, :512]).astype(np.float64)
    exact = E4M3[e[0, :, :512]] * np.repeat(s.astype(np.float64), 128, axis=1)
    np.testing.assert_array_equal(vals, exact)
    np.testing.assert_array_equal(out[:, 512:], e[0, :, 528:656].view("<u2"))


# --------------------------------------------------------------------------
# per-head NVFP4 cache
# --------------------------------------------------------------------------

def per_head_positions(page, side, off, h, bs, H, D):
    """Byte ranges of (page, side, off, h) under the format spec's reading of
    [K_data | K_scale | V_data | V_scale]: data [bs][H][D/2] then scales
    [bs][H][D/16] inside each side's bs * H * full_dim region."""
    g = {k: int(v) for k, v in ind.read_golden("entry_layout.txt")}
    fd = g[f"full_dim_{D}"]
    dd, sd = g[f"data_dim_{fd}"], g[f"scale_dim_{fd}"]
    region = bs * H * fd
    base = (page * 2 + side) * region
    data = base + (off * H + h) * dd
    scale = base + bs * H * dd + (off * H + h) * sd
    return slice(data, data + dd), slice(scale, scale + sd)


def test_per_head_write_matches_restatement(oracle_mod):
    w = wl.make_per_head("ph", 40, 4, 128, 6, 16, 3, 41, k_scale=1.0, v_scale=0.5)
    key, val, slots = wl.bf16_bits(w.key), wl.bf16_bits(w.value), wl.host(w.slot_mapping)
    fd = oracle_mod.nvfp4_full_dim(128)
    cache0 = wl.random_bytes((6, 2, 16, 4, fd), 3)
    cache = cache0.copy()
    assert oracle_mod.reshape_and_cache_nvfp4(key, val, slots, cache, 1.0, 0.5) == 0
    flat = cache.reshape(-1)
    touched = np.zeros(flat.size, bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        for side, (src, sc) in enumerate(((key, 1.0), (val, 0.5))):
            y = (ind.bf16_to_f32(src[t]) * (np.float32(1.0) / np.float32(sc))).astype(np.float32)
            packed, sf = ref_nvfp4_groups(y)
            for h in range(4):
                ds, ss = per_head_positions(s // 16, side, s % 16, h, 16, 4, 128)
                np.testing.assert_array_equal(flat[ds], packed[h])
                np.testing.assert_array_equal(flat[ss], sf[h])
                touched[ds] = touched[ss] = True
    np.testing.assert_array_equal(flat[~touched], cache0.reshape(-1)[~touched])


def test_per_head_dequant_round_trip(oracle_mod):
    for D in (64, 128, 256):
        w = wl.make_per_head("ph", 30, 2, D, 4, 16, 2, 42 + D, k_scale=2.0, v_scale=0.25)
        key, val, slots = wl.bf16_bits(w.key), wl.bf16_bits(w.value), wl.host(w.slot_mapping)
        cache = np.zeros((4, 2, 16, 2, oracle_mod.nvfp4_full_dim(D)), np.uint8)
        oracle_mod.reshape_and_cache_nvfp4(key, val, slots, cache, 2.0, 0.25)
        ko, vo, skipped = oracle_mod.dequant_nvfp4_per_head(cache, slots, 2, D, 2.0, 0.25)
        assert skipped == 0
        for src, out, sc in ((key, ko, 2.0), (val, vo, 0.25)):
            v = slots >= 0
            x = ind.bf16_to_f32(src[v]).astype(np.float64)
            y = (ind.bf16_to_f32(src[v]) * (np.float32(1) / np.float32(sc))).astype(np.float32)
            packed, sf = ref_nvfp4_groups(y)
            q = (E2M1[ind.unpack_e2m1(packed)] * np.repeat(E4M3[sf], 16, axis=-1)).astype(np.float32)
            want = ind.torch_bf16_bits(torch.from_numpy((q * np.float32(sc)).astype(np.float32)))
            np.testing.assert_array_equal(out[v], want)
            sfv = np.repeat(E4M3[sf], 16, axis=-1) * sc
            assert np.all(np.abs(ind.bf16_to_f32(out[v]) - x) <= 1.5 * sfv + np.abs(x) * 2.0 ** -8)
            assert np.all(out[~v] == 0)


# --------------------------------------------------------------------------
# sparse-decode index conversion
# --------------------------------------------------------------------------

def test_req_index_conversion_bruteforce(oracle_mod):
    g = np.random.Generator(np.random.PCG64(51))
    table, _, _, _ = wl.make_gather_batch(64, 16, [100, 37, 200, 5], [0, 0, 0, 0], 51)
    N, topk = 12, 8
    req = g.integers(0, 4, size=N).astype(np.int32)
    lens = np.array([100, 37, 200, 5])
    idx = (g.random((N, topk)) * lens[req][:, None]).astype(np.int32)
    idx[g.random((N, topk)) < 0.2] = -1
    out, skipped = oracle_mod.req_index_to_global_slot(req, idx, table, 16, 64)
    assert skipped == 0
    for i in range(N):
        for k in range(topk):
            p = idx[i, k]
            want = -1 if p < 0 else table[req[i], p // 16] * 16 + p % 16
            assert out[i, k] == want
    with pytest.raises(ValueError):
        oracle_mod.req_index_to_global_slot(req[:-1], idx, table, 16, 64)


def test_per_head_hnd_is_the_nhd_rows_permuted(oracle_mod):
    """The two layouts hold the same data and scale rows per (page, side):
    row (offset, head) sits at offset * H + head (NHD) or head * block_size
    + offset (HND)."""
    P, bs, H, D = 6, 16, 4, 128
    w = wl.make_per_head("lay", 70, H, D, P, bs, 4, 45, k_scale=0.5, v_scale=2.0)
    key, val, slots = wl.bf16_bits(w.key), wl.bf16_bits(w.value), wl.host(w.slot_mapping)
    fd = oracle_mod.nvfp4_full_dim(D)
    nhd = np.zeros((P, 2, bs, H, fd), np.uint8)
    hnd = np.zeros((P, 2, H, bs, fd), np.uint8)
    oracle_mod.reshape_and_cache_nvfp4(key, val, slots, nhd, 0.5, 2.0, layout="NHD")
    oracle_mod.reshape_and_cache_nvfp4(key, val, slots, hnd, 0.5, 2.0, layout="HND")
    dd, sd = D // 2, D // 16
    for p in range(P):
        for side in range(2):
            a, b = nhd[p, side].reshape(-1), hnd[p, side].reshape(-1)
            ad, as_ = a[:bs * H * dd].reshape(bs, H, dd), a[bs * H * dd:].reshape(bs, H, sd)
            bd, bs_ = b[:bs * H * dd].reshape(H, bs, dd), b[bs * H * dd:].reshape(H, bs, sd)
            np.testing.assert_array_equal(ad, bd.transpose(1, 0, 2))
            np.testing.assert_array_equal(as_, bs_.transpose(1, 0, 2))
    k1, v1, _ = oracle_mod.dequant_nvfp4_per_head(nhd, slots, H, D, 0.5, 2.0, layout="NHD")
    k2, v2, _ = oracle_mod.dequant_nvfp4_per_head(hnd, slots, H, D, 0.5, 2.0, layout="HND")
    np.testing.assert_array_equal(k1, k2)
    np.testing.assert_array_equal(v1, v2)
