"""Pins for the oracle's sparse MLA attention over the nvfp4_ds_mla and
fp8_ds_mla caches.

The attention is a plain definition (softmax-weighted sum of the cached latent
rows, MQA form), so the oracle is pinned against an independent float64
evaluation of that definition in numpy on keys whose values are known by
construction, plus the special cases the definition fixes: one valid entry,
duplicated and permuted lists, unused and out-of-range entries, empty lists
and large scores."""
import numpy as np
import pytest

BS = 16


def bf16_bits_of(x):
    """bf16 bit patterns (round toward zero) of float32 values, and the values."""
    bits = (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    return bits, (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def exact_keys(n, seed, oracle_mod):
    """n latent rows whose nvfp4_ds_mla encoding is exact: each NoPE group is
    c * S with e2m1 codes c (max |c| = 6) and an e4m3 scale S; RoPE values are
    e4m3 values.  Returns (kv_c bits, k_pe bits, exact float64 keys [n, 576])."""
    g = np.random.Generator(np.random.PCG64(seed))
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    e4m3 = np.array([oracle_mod.e4m3_value(c) for c in range(0x08, 0x70)])   # normal, positive
    keys = np.zeros((n, 576))
    for i in range(n):
        for grp in range(32):
            c = mags[g.integers(0, 8, 16)] * np.where(g.random(16) < 0.5, -1, 1)
            c[g.integers(0, 16)] = 6.0 * (1 if g.random() < 0.5 else -1)
            keys[i, 16 * grp:16 * grp + 16] = c * e4m3[g.integers(0, len(e4m3))]
        keys[i, 512:] = e4m3[g.integers(0, len(e4m3), 64)] * np.where(g.random(64) < 0.5, -1, 1)
    kv_c, _ = bf16_bits_of(keys[:, :512])
    k_pe, _ = bf16_bits_of(keys[:, 512:])
    return kv_c, k_pe, keys


def build_cache(oracle_mod, n_slots, seed, num_blocks=8):
    """A cache whose first n_slots slots (in a seeded order) hold exact keys."""
    kv_c, k_pe, keys = exact_keys(n_slots, seed, oracle_mod)
    g = np.random.Generator(np.random.PCG64(seed + 1))
    slots = g.permutation(num_blocks * BS)[:n_slots].astype(np.int64)
    cache = np.zeros((num_blocks, BS, 352), np.uint8)
    assert oracle_mod.write_nvfp4_ds_mla(kv_c, k_pe, slots, cache) == 0
    return cache, slots, keys


def numpy_attention(q, keys, scale):
    """float64 softmax attention of q [H, 576] over keys [n, 576], values
    keys[:, :512]: (o [H, 512], lse [H])."""
    s = scale * (q @ keys.T)
    m = s.max(axis=1, keepdims=True)
    w = np.exp(s - m)
    lse = (m[:, 0] + np.log(w.sum(axis=1)))
    return (w @ keys[:, :512]) / w.sum(axis=1, keepdims=True), lse


def random_q(T, H, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    return bf16_bits_of(g.standard_normal((T, H, 576)).astype(np.float32))


def test_encoding_of_the_keys_is_exact(oracle_mod):
    cache, slots, keys = build_cache(oracle_mod, 20, 7)
    for i, s in enumerate(slots):
        np.testing.assert_array_equal(oracle_mod.decode_nvfp4_ds_mla_entry(cache[s // BS, s % BS]), keys[i])


@pytest.mark.parametrize("scale", [1.0 / 24.0, 0.2, 3.0])
def test_attention_matches_numpy_definition(oracle_mod, scale):
    """Several tokens, several heads, each with its own slot list (with unused
    entries), against numpy's float64 evaluation on the exact keys."""
    cache, slots, keys = build_cache(oracle_mod, 60, 11)
    T, H, topk = 5, 6, 24
    qb, qv = random_q(T, H, 12)
    g = np.random.Generator(np.random.PCG64(13))
    idx = np.full((T, topk), -1, np.int32)
    for t in range(T):
        pick = g.choice(60, size=topk - 3 * t, replace=False)
        idx[t, :len(pick)] = slots[pick]
        g.shuffle(idx[t])
    o, lse, skipped = oracle_mod.sparse_mla_attention_nvfp4_ds_mla(qb, idx, cache, scale)
    assert skipped == 0
    slot_row = {int(s): i for i, s in enumerate(slots)}
    for t in range(T):
        rows = [slot_row[int(s)] for s in idx[t] if s >= 0]
        want_o, want_lse = numpy_attention(qv[t], keys[rows], scale)
        np.testing.assert_allclose(o[t], want_o, rtol=1e-11, atol=1e-11 * np.abs(keys).max())
        np.testing.assert_allclose(lse[t], want_lse, rtol=1e-12, atol=1e-12)


def test_single_valid_entry_returns_its_value(oracle_mod):
    cache, slots, keys = build_cache(oracle_mod, 4, 21)
    qb, qv = random_q(1, 3, 22)
    idx = np.array([[-1, slots[2], -1, -1]], np.int32)
    o, lse, _ = oracle_mod.sparse_mla_attention_nvfp4_ds_mla(qb, idx, cache, 0.5)
    for h in range(3):
        np.testing.assert_array_equal(o[0, h], keys[2, :512])
        assert lse[0, h] == pytest.approx(0.5 * float(qv[0, h] @ keys[2]), rel=1e-14, abs=1e-14)


def test_duplicated_and_permuted_lists(oracle_mod):
    """Listing every slot twice adds log 2 to lse and leaves o unchanged;
    permuting the list changes nothing but the summation order."""
    cache, slots, keys = build_cache(oracle_mod, 16, 31)
    qb, _ = random_q(1, 4, 32)
    base = slots[:10].astype(np.int32)[None, :]
    twice = np.concatenate([base, base], axis=1)
    perm = base[:, np.random.Generator(np.random.PCG64(33)).permutation(10)]
    o1, l1, _ = oracle_mod.sparse_mla_attention_nvfp4_ds_mla(qb, base, cache, 0.3)
    o2, l2, _ = oracle_mod.sparse_mla_attention_nvfp4_ds_mla(qb, twice, cache, 0.3)
    o3, l3, _ = oracle_mod.sparse_mla_attention_nvfp4_ds_mla(qb, perm, cache, 0.3)
    np.testing.assert_allclose(l2, l1 + np.log(2.0), rtol=0, atol=1e-12)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l3, l1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o3, o1, rtol=1e-12, atol=1e-12)


def test_unused_and_out_of_range_entries_are_ignored(oracle_mod):
    cache, slots, keys = build_cache(oracle_mod, 8, 41)
    qb, _ = random_q(1, 2, 42)
    clean = slots[:6].astype(np.int32)[None, :]
    noisy = np.array([[clean[0, 0], -1, 8 * BS, clean[0, 1], clean[0, 2], -7, clean[0, 3],
                       1 << 30, clean[0, 4], clean[0, 5]]], np.int32)
    o1, l1, s1 = oracle_mod.sparse_mla_attention_nvfp4_ds_mla(qb, clean, cache, 0.25)
    o2, l2, s2 = oracle_mod.sparse_mla_attention_nvfp4_ds_mla(qb, noisy, cache, 0.25)
    assert (s1, s2) == (0, 2)
    np.testing.assert_array_equal(o2, o1)
    np.testing.assert_array_equal(l2, l1)


def test_empty_lists_give_zero_output_and_minus_infinity(oracle_mod):
    cache, _, _ = build_cache(oracle_mod, 4, 51)
    qb, _ = random_q(2, 3, 52)
    o, lse, _ = oracle_mod.sparse_mla_attention_nvfp4_ds_mla(qb, np.full((2, 5), -1, np.int32), cache, 1.0)
    assert not o.any() and np.all(np.isneginf(lse))
    o, lse, _ = oracle_mod.sparse_mla_attention_nvfp4_ds_mla(qb, np.zeros((2, 0), np.int32), cache, 1.0)
    assert not o.any() and np.all(np.isneginf(lse))


def test_large_scores_do_not_overflow(oracle_mod):
    """Scores in the thousands: the max-subtracted form stays finite and
    matches numpy's."""
    cache, slots, keys = build_cache(oracle_mod, 12, 61)
    qb, qv = random_q(1, 2, 62)
    idx = slots[:12].astype(np.int32)[None, :]
    o, lse, _ = oracle_mod.sparse_mla_attention_nvfp4_ds_mla(qb, idx, cache, 40.0)
    want_o, want_lse = numpy_attention(qv[0], keys[:12], 40.0)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)) and np.abs(want_lse).max() > 1000
    np.testing.assert_allclose(o[0], want_o, rtol=1e-9, atol=1e-9 * np.abs(keys).max())
    np.testing.assert_allclose(lse[0], want_lse, rtol=1e-12)


# --------------------------------------------------------------------------
# the same consumer over the 656-byte fp8_ds_mla cache
# --------------------------------------------------------------------------

def exact_fp8_cache(oracle_mod, n_slots, seed, num_blocks=8):
    """Entries built byte by byte whose upconvert is exact: e4m3 NoPE codes
    with power-of-two tile scales, bf16 RoPE.  Returns (cache, slots, keys)."""
    g = np.random.Generator(np.random.PCG64(seed))
    cache = np.zeros((num_blocks, BS, 656), np.uint8)
    slots = g.permutation(num_blocks * BS)[:n_slots]
    keys = np.zeros((n_slots, 576))
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    for i, s in enumerate(slots):
        e = cache[s // BS, s % BS]
        codes = finite[g.integers(0, len(finite), 512)]
        scales = (2.0 ** g.integers(-6, 4, 4)).astype(np.float32)
        e[:512] = codes
        e[512:528] = np.frombuffer(scales.astype("<f4").tobytes(), np.uint8)
        rope_bits, rope = bf16_bits_of(g.standard_normal(64).astype(np.float32))
        e[528:656] = np.frombuffer(rope_bits.astype("<u2").tobytes(), np.uint8)
        keys[i, :512] = [oracle_mod.e4m3_value(int(c)) * float(scales[k // 128]) for k, c in enumerate(codes)]
        keys[i, 512:] = rope
    return cache, slots, keys


def test_fp8_entry_decode_is_exact_on_constructed_entries(oracle_mod):
    cache, slots, keys = exact_fp8_cache(oracle_mod, 6, 71)
    for i, s in enumerate(slots):
        np.testing.assert_array_equal(oracle_mod.decode_fp8_ds_mla_entry(cache[s // BS, s % BS]), keys[i])


@pytest.mark.parametrize("scale", [1.0 / 24.0, 0.15])
def test_fp8_attention_matches_numpy_definition(oracle_mod, scale):
    cache, slots, keys = exact_fp8_cache(oracle_mod, 40, 72)
    T, H, topk = 4, 5, 20
    qb, qv = random_q(T, H, 73)
    g = np.random.Generator(np.random.PCG64(74))
    idx = np.full((T, topk), -1, np.int32)
    for t in range(T):
        pick = g.choice(40, size=topk - 2 * t, replace=False)
        idx[t, :len(pick)] = slots[pick]
    o, lse, skipped = oracle_mod.sparse_mla_attention_fp8_ds_mla(qb, idx, cache, scale)
    assert skipped == 0
    slot_row = {int(s): i for i, s in enumerate(slots)}
    for t in range(T):
        rows = [slot_row[int(s)] for s in idx[t] if s >= 0]
        want_o, want_lse = numpy_attention(qv[t], keys[rows], scale)
        np.testing.assert_allclose(o[t], want_o, rtol=1e-11, atol=1e-11 * np.abs(keys).max())
        np.testing.assert_allclose(lse[t], want_lse, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# dense prefill: every context position of a request, read through its
# block-table row (vLLM PR #48642, "Function and motivation",
# _compute_prefill_context)
# ---------------------------------------------------------------------------

def prefill_case(oracle_mod, seed, ctx_lens, q_lens, H, num_blocks=12):
    """Requests whose contexts hold exact keys: request b's positions p <
    ctx_lens[b] live at entry p % BS of block table[b][p // BS] (distinct
    shuffled blocks).  Returns (cache, table, query_start, keys per request,
    q bits, q values)."""
    g = np.random.Generator(np.random.PCG64(seed))
    n_blk = [(c + BS - 1) // BS for c in ctx_lens]
    order = g.permutation(num_blocks)
    assert sum(n_blk) <= num_blocks
    width = max(1, max(n_blk))
    table = np.full((len(ctx_lens), width), -1, np.int32)
    cache = np.zeros((num_blocks, BS, 352), np.uint8)
    keys, used = [], 0
    for b, c in enumerate(ctx_lens):
        table[b, :n_blk[b]] = order[used:used + n_blk[b]]
        used += n_blk[b]
        kv_c, k_pe, k = exact_keys(c, seed + 10 + b, oracle_mod)
        slots = np.array([table[b, p // BS] * BS + p % BS for p in range(c)], np.int64)
        if c:
            assert oracle_mod.write_nvfp4_ds_mla(kv_c, k_pe, slots, cache) == 0
        keys.append(k)
    qs = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    qb, qv = random_q(int(qs[-1]), H, seed + 5)
    return cache, table, qs, keys, qb, qv


@pytest.mark.parametrize("scale", [1.0 / 24.0, 0.7])
def test_prefill_matches_numpy_definition(oracle_mod, scale):
    """Three requests (ragged contexts across block boundaries, 1-3 query
    tokens each) against numpy's float64 evaluation on the exact keys."""
    ctx, ql, H = [37, 16, 50], [2, 1, 3], 5
    cache, table, qs, keys, qb, qv = prefill_case(oracle_mod, 41, ctx, ql, H)
    o, lse, skipped = oracle_mod.prefill_mla_attention_nvfp4_ds_mla(qb, qs, ctx, table, cache, scale)
    assert skipped == 0
    for b in range(3):
        for t in range(qs[b], qs[b + 1]):
            want_o, want_lse = numpy_attention(qv[t], keys[b], scale)
            np.testing.assert_allclose(o[t], want_o, rtol=1e-11, atol=1e-11 * np.abs(keys[b]).max())
            np.testing.assert_allclose(lse[t], want_lse, rtol=1e-12, atol=1e-12)


def test_prefill_is_independent_of_block_placement(oracle_mod):
    """Moving a request's blocks elsewhere in the cache (the table updated
    with them) changes nothing: the context is addressed only through the
    table."""
    ctx, ql, H = [40, 23], [2, 2], 3
    cache, table, qs, _, qb, _ = prefill_case(oracle_mod, 51, ctx, ql, H)
    perm = np.random.Generator(np.random.PCG64(52)).permutation(cache.shape[0])
    moved = np.empty_like(cache)
    moved[perm] = cache                              # block i -> perm[i]
    table2 = np.where(table >= 0, perm[np.maximum(table, 0)], -1).astype(np.int32)
    o1, l1, _ = oracle_mod.prefill_mla_attention_nvfp4_ds_mla(qb, qs, ctx, table, cache, 0.3)
    o2, l2, _ = oracle_mod.prefill_mla_attention_nvfp4_ds_mla(qb, qs, ctx, table2, moved, 0.3)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_prefill_empty_context_bad_blocks_and_no_queries(oracle_mod):
    """A request with no context gives o = 0 and lse = -inf; positions whose
    block id or table column is out of range are skipped and counted (the
    rest still attend); a request with no query tokens writes nothing."""
    ctx, ql, H = [0, 30, 20], [2, 1, 0], 2
    cache, table, qs, keys, qb, qv = prefill_case(oracle_mod, 61, ctx, ql, H)
    table = table.copy()
    table[1, 1] = 99                                 # positions 16..29 of request 1: bad block id
    ctx2 = np.array([0, 30, 20], np.int32)
    o, lse, skipped = oracle_mod.prefill_mla_attention_nvfp4_ds_mla(qb, qs, ctx2, table, cache, 0.5)
    assert skipped == 14
    assert not o[0:2].any() and np.all(np.isneginf(lse[0:2]))
    want_o, want_lse = numpy_attention(qv[2], keys[1][:16], 0.5)
    np.testing.assert_allclose(o[2], want_o, rtol=1e-11, atol=1e-11 * np.abs(keys[1]).max())
    np.testing.assert_allclose(lse[2], want_lse, rtol=1e-12, atol=1e-12)
    wide = np.array([0, 40, 20], np.int32)           # 40 positions: columns past the table width
    _, _, skipped = oracle_mod.prefill_mla_attention_nvfp4_ds_mla(qb, qs, wide, table, cache, 0.5)
    assert skipped == (32 - 16) + (40 - 32)          # bad block: positions 16..31; past the width: 32..39


def test_prefill_fp8_matches_numpy_definition(oracle_mod):
    """The fp8_ds_mla form: entries of e4m3 codes with power-of-two tile
    scales and bf16 RoPE (exact by construction), two requests."""
    g = np.random.Generator(np.random.PCG64(71))
    nb = 6
    cache = np.zeros((nb, BS, 656), np.uint8)
    codes = g.integers(0, 0x7f, (nb, BS, 512)).astype(np.uint8) | (g.integers(0, 2, (nb, BS, 512)) << 7).astype(np.uint8)
    codes[(codes & 0x7f) == 0x7f] = 0x10
    cache[:, :, :512] = codes
    scales = (2.0 ** g.integers(-4, 5, (nb, BS, 4))).astype("<f4")
    cache[:, :, 512:528] = scales.view(np.uint8).reshape(nb, BS, 16)
    rope_bits, rope = bf16_bits_of(g.standard_normal((nb, BS, 64)).astype(np.float32))
    cache[:, :, 528:656] = rope_bits.astype("<u2").view(np.uint8).reshape(nb, BS, 128)
    e4 = np.array([oracle_mod.e4m3_value(c) for c in range(256)])
    dec = np.concatenate([e4[codes] * np.repeat(scales.astype(np.float64), 128, axis=2), rope], axis=2)
    table = np.array([[4, 1, 0], [2, 5, -1]], np.int32)
    ctx = np.array([40, 17], np.int32)
    qs = np.array([0, 2, 3], np.int32)
    qb, qv = random_q(3, 4, 72)
    o, lse, skipped = oracle_mod.prefill_mla_attention_fp8_ds_mla(qb, qs, ctx, table, cache, 0.02)
    assert skipped == 0
    for b in range(2):
        k = np.stack([dec[table[b, p // BS], p % BS] for p in range(ctx[b])])
        for t in range(qs[b], qs[b + 1]):
            want_o, want_lse = numpy_attention(qv[t], k, 0.02)
            np.testing.assert_allclose(o[t], want_o, rtol=1e-11, atol=1e-11 * np.abs(k).max())
            np.testing.assert_allclose(lse[t], want_lse, rtol=1e-12, atol=1e-12)
