"""GPU parity of the sparse MLA attention read straight from the nvfp4_ds_mla
cache, against the oracle's float64 evaluation.

The output is floating point, so the bar is a tolerance derived from the
kernel's arithmetic (the decoded keys are exact in both):
  * scores: fp32 accumulation of 576 exact bf16 products, error at most
    e_s = 576 * 2^-24 * scale * max_j sum_d |q_d| |k_jd|  (per token and head);
  * weights: exp in fp32 then rounded to bf16 (relative 2^-9), and the
    denominator sums the rounded weights, so each normalised weight carries a
    relative error of at most eps = 2^-9 + e_s + 2^-20;
  * a convex combination whose weights move by a relative eps moves by at
    most 2 eps / (1 - eps) * max_j |v_j|; the fp32 accumulation of P V adds
    far less, and the bf16 output rounding adds 2^-9 |o|;
  * lse moves by at most eps + e_s, plus fp32 rounding of the result.
The bound is checked per element with vmax = max_j |v_j| of the token's
valid slots.
"""
import numpy as np
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


@pytest.fixture(scope="module")
def threads(oracle_mod):
    return oracle_mod.default_threads()


# entry format -> (entry bytes, oracle write, oracle decode, oracle attention, kernel entry point)
FORMATS = {
    "nvfp4": (352, "write_nvfp4_ds_mla", "decode_nvfp4_ds_mla_entry", "sparse_mla_attention_nvfp4_ds_mla",
              "kvq_sparse_mla_attention_nvfp4_ds_mla"),
    "fp8": (656, "write_fp8_ds_mla", "decode_fp8_ds_mla_entry", "sparse_mla_attention_fp8_ds_mla",
            "kvq_sparse_mla_attention_fp8_ds_mla"),
}


def host_cache(oracle_mod, fill, threads=1, fmt="nvfp4"):
    entry, write = FORMATS[fmt][:2]
    cache = np.zeros((fill.num_blocks, fill.block_size, entry), np.uint8)
    assert getattr(oracle_mod, write)(wl.bf16_bits(fill.kv_c), wl.bf16_bits(fill.k_pe),
                                      wl.host(fill.slot_mapping), cache, threads=threads) == 0
    return cache


def decoded_keys(oracle_mod, cache, slots):
    """float64 [n, 576] decoded entries of the given slots (oracle decode)."""
    bs = cache.shape[1]
    decode = getattr(oracle_mod, "decode_fp8_ds_mla_entry" if cache.shape[2] == 656 else
                     "decode_nvfp4_ds_mla_entry")
    uniq, inv = np.unique(slots, return_inverse=True)
    table = np.stack([decode(cache[s // bs, s % bs]) for s in uniq])
    return table[inv]


def q_values(q):
    bits = wl.bf16_bits(q).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


def check(oracle_mod, cache, q, idx, scale, out, lse, threads=1, tokens=None):
    """Compares GPU out / lse with the oracle on the given tokens (all by default)."""
    qb = wl.bf16_bits(q)
    idx = np.asarray(idx, np.int32)
    tokens = np.arange(q.shape[0]) if tokens is None else np.asarray(tokens)
    attention = getattr(oracle_mod, FORMATS["fp8" if cache.shape[2] == 656 else "nvfp4"][3])
    want_o, want_lse, _ = attention(np.ascontiguousarray(qb[tokens]), idx[tokens], cache, scale, threads=threads)
    got_o = out.float().cpu().numpy()[tokens].astype(np.float64)
    got_lse = lse.cpu().numpy()[tokens].astype(np.float64)
    qv = q_values(q)[tokens]
    n_slots = cache.shape[0] * cache.shape[1]
    for i, t in enumerate(tokens):
        valid = idx[t][(idx[t] >= 0) & (idx[t] < n_slots)]
        if valid.size == 0:
            assert not np.any(got_o[i]), f"token {t}: no valid slot but nonzero output"
            assert np.all(np.isneginf(got_lse[i])), f"token {t}: lse {got_lse[i]}"
            continue
        keys = decoded_keys(oracle_mod, cache, valid)
        vmax = np.abs(keys[:, :512]).max()
        e_s = 576 * 2.0 ** -24 * abs(scale) * (np.abs(qv[i]) @ np.abs(keys).T).max(axis=1)   # [H]
        eps = 2.0 ** -9 + e_s + 2.0 ** -20
        tol_o = (2 * eps / (1 - eps))[:, None] * vmax + 2.0 ** -9 * np.abs(want_o[i]) + 1e-30
        err_o = np.abs(got_o[i] - want_o[i])
        bad = err_o > tol_o
        assert not bad.any(), (f"token {t}: {int(bad.sum())} outputs beyond the bound; worst "
                               f"{float((err_o / tol_o).max()):.3f} x bound")
        tol_l = eps + e_s + 2.0 ** -22 * np.abs(want_lse[i])
        err_l = np.abs(got_lse[i] - want_lse[i])
        assert np.all(err_l <= tol_l), f"token {t}: lse error {err_l.max()} > {tol_l.min()}"


def run(kvq, oracle_mod, w, cache=None, threads=1, tokens=None, strided=False, fmt="nvfp4"):
    if cache is None:
        cache = host_cache(oracle_mod, w.fill, threads, fmt)
    dcache = torch.from_numpy(cache).to(DEV)
    q = w.q.to(DEV)
    T, H = q.shape[0], q.shape[1]
    if strided:      # q rows and out rows inside wider buffers
        qbig = torch.zeros((T, H, 640), dtype=torch.bfloat16, device=DEV)
        qbig[:, :, 32:608] = q
        q = qbig[:, :, 32:608]
        obig = torch.full((T, H, 520), -7.0, dtype=torch.bfloat16, device=DEV)
        out = obig[:, :, 8:520]
        lbig = torch.full((T, H + 5), -7.0, dtype=torch.float32, device=DEV)
        lse = lbig[:, :H]
    else:
        out = torch.full((T, H, 512), -7.0, dtype=torch.bfloat16, device=DEV)
        lse = torch.full((T, H), -7.0, dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    idx = w.indices.to(DEV)
    getattr(kvq, FORMATS[fmt][4])(q, idx, dcache, w.softmax_scale, out=out, lse=lse, status=status)
    torch.cuda.synchronize()
    check(oracle_mod, cache, w.q, wl.host(w.indices), w.softmax_scale, out, lse, threads, tokens)
    if strided:
        assert torch.all(obig[:, :, :8] == -7.0) and torch.all(lbig[:, H:] == -7.0)
    return int(status.item())


CASES = [
    ("H128 top64", dict(num_tokens=3, num_heads=128, topk=64, num_blocks=8, block_size=64, seed=301)),
    ("H16 top100 ragged", dict(num_tokens=5, num_heads=16, topk=100, num_blocks=8, block_size=64, seed=302,
                               p_unused=0.2)),
    ("H1 top33", dict(num_tokens=4, num_heads=1, topk=33, num_blocks=4, block_size=16, seed=303)),
    ("H64 top256 sharp", dict(num_tokens=3, num_heads=64, topk=256, num_blocks=16, block_size=64, seed=304,
                              softmax_scale=0.25)),
    ("H128 top512 q x4", dict(num_tokens=2, num_heads=128, topk=512, num_blocks=16, block_size=64, seed=305,
                              q_scale=4.0, p_unused=0.5)),
    ("H96 top31", dict(num_tokens=6, num_heads=96, topk=31, num_blocks=4, block_size=32, seed=306)),
    # three full tiles: the score and receive double buffers wrap, the K ring fills
    ("H128 top192", dict(num_tokens=2, num_heads=128, topk=192, num_blocks=8, block_size=64, seed=307)),
]


@pytest.mark.parametrize("fmt", sorted(FORMATS))
@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_attention_parity(kvq, oracle_mod, name, kw, fmt):
    w = wl.make_attention(name, **kw)
    assert run(kvq, oracle_mod, w, fmt=fmt) == 0


@pytest.mark.parametrize("fmt", sorted(FORMATS))
def test_attention_strided_q_out_lse(kvq, oracle_mod, fmt):
    w = wl.make_attention("strided", 3, 20, 70, 8, 64, 311, p_unused=0.1)
    assert run(kvq, oracle_mod, w, strided=True, fmt=fmt) == 0


@pytest.mark.parametrize("fmt", sorted(FORMATS))
def test_attention_empty_and_bad_slots(kvq, oracle_mod, fmt):
    """Token 0: every entry unused; token 1: only out-of-range slots; token 2:
    a mix; topk = 40.  Out-of-range slots set the status bit and are skipped."""
    w = wl.make_attention("edge", 3, 8, 40, 4, 16, 312)
    idx = wl.host(w.indices).copy()
    idx[0] = -1
    idx[1] = 64 + np.arange(40)
    idx[2, ::3] = 1 << 30
    w.indices = torch.from_numpy(idx)
    assert run(kvq, oracle_mod, w, fmt=fmt) == kvq.STATUS_BAD_INDEX


def test_attention_topk_zero(kvq, oracle_mod):
    w = wl.make_attention("topk0", 4, 8, 0, 4, 16, 313)
    assert run(kvq, oracle_mod, w) == 0


def test_attention_duplicate_slots(kvq, oracle_mod):
    w = wl.make_attention("dup", 2, 32, 64, 4, 16, 314)
    idx = wl.host(w.indices).copy()
    idx[:, 32:] = idx[:, :32]
    w.indices = torch.from_numpy(idx)
    assert run(kvq, oracle_mod, w) == 0


def test_attention_full_size_sampled(kvq, oracle_mod, threads):
    """The benchmark's decode workload (4096 tokens x 128 heads, top-2048 over
    a 65536 x 64 cache, 10 % unused) in one launch; 48 sampled tokens (first,
    last, random) against the oracle."""
    fill = wl.make_fill("attention fill", 65536, 64, 1006, DEV, rng="device")
    cache_host = host_cache(oracle_mod, fill, threads)       # the oracle's own write
    cache = torch.from_numpy(cache_host).to(DEV)
    w = wl.sparse_attention(DEV, fill=fill)
    del fill
    out, lse = kvq.kvq_sparse_mla_attention_nvfp4_ds_mla(w.q, w.indices, cache, w.softmax_scale)
    torch.cuda.synchronize()
    g = np.random.Generator(np.random.PCG64(77))
    tokens = np.unique(np.concatenate([[0, w.num_tokens - 1], g.choice(w.num_tokens, 46, replace=False)]))
    check(oracle_mod, cache_host, w.q, wl.host(w.indices), w.softmax_scale, out, lse, threads, tokens)


def test_attention_random_cache_bytes(kvq, oracle_mod):
    """Every e2m1 code, negative and subnormal scale bytes and large RoPE
    values: a cache of random bytes (the two e4m3 NaN codes replaced)."""
    cache = wl.random_bytes((16, 64, 352), 321)
    wl.nan_free_e4m3_bytes(cache[:, :, 256:])          # RoPE and scale bytes
    w = wl.make_attention("random bytes", 4, 128, 192, 16, 64, 322, p_unused=0.1, softmax_scale=0.01)
    assert run(kvq, oracle_mod, w, cache=cache) == 0


def test_attention_single_token_strided_indices_no_lse(kvq, oracle_mod):
    """One token (one cluster), top-k slots taken from a wider index tensor,
    and no lse output (the output alone is still checked)."""
    w = wl.make_attention("one token", 1, 128, 160, 8, 64, 331, p_unused=0.15)
    cache = host_cache(oracle_mod, w.fill)
    wide = torch.full((1, 160 + 24), 5, dtype=torch.int32)
    wide[:, :160] = w.indices
    idx = wide.to(DEV)[:, :160]
    out = torch.full((1, 128, 512), -7.0, dtype=torch.bfloat16, device=DEV)
    kvq.kvq_sparse_mla_attention_nvfp4_ds_mla(w.q.to(DEV), idx, torch.from_numpy(cache).to(DEV), w.softmax_scale,
                                              out=out, lse=False)
    torch.cuda.synchronize()
    _, lse_ref, _ = oracle_mod.sparse_mla_attention_nvfp4_ds_mla(wl.bf16_bits(w.q), wl.host(w.indices), cache,
                                                                 w.softmax_scale)
    check(oracle_mod, cache, w.q, wl.host(w.indices), w.softmax_scale, out,
          torch.from_numpy(lse_ref.astype(np.float32)))


def test_attention_fp8_random_codes_and_scales(kvq, oracle_mod):
    """fp8_ds_mla entries of random bytes: every e4m3 code (NaN codes
    replaced), power-of-two tile scales from 2^-8 to 2^8 and bf16 RoPE values
    of magnitudes 2^-8 .. 2^8 (scores must fit the fp32 accumulator, as
    for any input of the kernel)."""
    g = np.random.Generator(np.random.PCG64(341))
    cache = wl.random_bytes((16, 64, 656), 342)
    wl.nan_free_e4m3_bytes(cache[:, :, :512])
    scales = (2.0 ** g.integers(-8, 9, (16, 64, 4))).astype("<f4")
    cache[:, :, 512:528] = scales.view(np.uint8).reshape(16, 64, 16)
    rope = (g.standard_normal((16, 64, 64)) * 2.0 ** g.integers(-8, 9, (16, 64, 64))).astype(np.float32)
    rope_bits = (rope.view(np.uint32) >> 16).astype("<u2")
    cache[:, :, 528:656] = rope_bits.view(np.uint8).reshape(16, 64, 128)
    w = wl.make_attention("fp8 random bytes", 4, 128, 192, 16, 64, 343, p_unused=0.1, softmax_scale=1e-4)
    assert run(kvq, oracle_mod, w, cache=cache, fmt="fp8") == 0


def test_attention_fp8_full_size_sampled(kvq, oracle_mod, threads):
    """4096 tokens x 128 heads, top-2048 over a 32768 x 64 fp8_ds_mla cache
    filled by the oracle's write; 32 sampled tokens against the oracle."""
    fill = wl.make_fill("fp8 attention fill", 32768, 64, 1004, DEV, entry_bytes=656, rng="device")
    cache_host = host_cache(oracle_mod, fill, threads, "fp8")
    cache = torch.from_numpy(cache_host).to(DEV)
    w = wl.make_attention("fp8 attention", 4096, 128, 2048, 32768, 64, 1008, DEV, p_unused=0.1, fill=fill,
                          rng="device")
    del fill
    out, lse = kvq.kvq_sparse_mla_attention_fp8_ds_mla(w.q, w.indices, cache, w.softmax_scale)
    torch.cuda.synchronize()
    g = np.random.Generator(np.random.PCG64(78))
    tokens = np.unique(np.concatenate([[0, w.num_tokens - 1], g.choice(w.num_tokens, 30, replace=False)]))
    check(oracle_mod, cache_host, w.q, wl.host(w.indices), w.softmax_scale, out, lse, threads, tokens)


@pytest.mark.parametrize("fmt", sorted(FORMATS))
@pytest.mark.parametrize("heads", [2, 32, 127])
@pytest.mark.parametrize("topk", [1, 65, 257])
def test_attention_shape_sweep(kvq, oracle_mod, fmt, heads, topk):
    """Head counts that are not a warp multiple and top-k lengths of one
    slot, one slot past a tile and one past four tiles."""
    w = wl.make_attention(f"sweep H{heads} k{topk}", 2, heads, topk, 8, 64, 400 + heads + topk, p_unused=0.05)
    assert run(kvq, oracle_mod, w, fmt=fmt) == 0


@pytest.mark.parametrize("fmt", sorted(FORMATS))
def test_attention_repeated_launches_bit_identical(kvq, oracle_mod, fmt):
    """The kernel fixes every accumulation order (the MMAs, the score
    exchange, the softmax sums), so repeated launches on the same inputs give
    the same bits; a race in the exchange or the buffer hand-offs would show
    as launch-to-launch differences.  152 tokens: one wave of clusters."""
    w = wl.make_attention("repeat", 152, 128, 512, 16, 64, 331, p_unused=0.1)
    cache = torch.from_numpy(host_cache(oracle_mod, w.fill, fmt=fmt)).to(DEV)
    q, idx = w.q.to(DEV), w.indices.to(DEV)
    fn = getattr(kvq, FORMATS[fmt][4])
    out0, lse0 = fn(q, idx, cache, w.softmax_scale)
    for _ in range(8):
        out, lse = fn(q, idx, cache, w.softmax_scale)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), out0.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), lse0.view(torch.int32))


# ---------------------------------------------------------------------------
# dense prefill: the query tokens of a request attend to its whole context
# through the block table; (token, head) rows are packed 128 to a CTA, so a
# CTA's decoded key tiles feed several query tokens when H < 128
# ---------------------------------------------------------------------------

PREFILL_FORMATS = {"nvfp4": ("prefill_mla_attention_nvfp4_ds_mla", "kvq_prefill_mla_attention_nvfp4_ds_mla"),
                   "fp8": ("prefill_mla_attention_fp8_ds_mla", "kvq_prefill_mla_attention_fp8_ds_mla")}


def check_prefill(oracle_mod, cache, w, out, lse, threads=1, requests=None):
    """GPU out / lse against the oracle's dense prefill for the given
    requests (all by default), within the bound of check()."""
    fmt = "fp8" if cache.shape[2] == 656 else "nvfp4"
    qs, ctx, table = wl.host(w.query_start), wl.host(w.context_lens), wl.host(w.block_table)
    qb = wl.bf16_bits(w.q)
    qv = q_values(w.q)
    got_o = out.float().cpu().numpy().astype(np.float64)
    got_lse = lse.cpu().numpy().astype(np.float64)
    bs, nb = cache.shape[1], cache.shape[0]
    requests = range(len(ctx)) if requests is None else requests
    for b in requests:
        sub_qs = np.array([0, qs[b + 1] - qs[b]], np.int32)
        if sub_qs[1] == 0:
            continue
        want_o, want_lse, _ = getattr(oracle_mod, PREFILL_FORMATS[fmt][0])(
            np.ascontiguousarray(qb[qs[b]:qs[b + 1]]), sub_qs, ctx[b:b + 1], table[b:b + 1], cache, w.softmax_scale,
            threads=threads)
        slots = [table[b, p // bs] * bs + p % bs for p in range(max(ctx[b], 0))
                 if p // bs < table.shape[1] and 0 <= table[b, p // bs] < nb]
        for i, t in enumerate(range(qs[b], qs[b + 1])):
            if not slots:
                assert not np.any(got_o[t]), f"request {b} token {t}: no context but nonzero output"
                assert np.all(np.isneginf(got_lse[t])), f"request {b} token {t}: lse {got_lse[t]}"
                continue
            keys = decoded_keys(oracle_mod, cache, np.asarray(slots))
            vmax = np.abs(keys[:, :512]).max()
            e_s = 576 * 2.0 ** -24 * abs(w.softmax_scale) * (np.abs(qv[t]) @ np.abs(keys).T).max(axis=1)
            eps = 2.0 ** -9 + e_s + 2.0 ** -20
            tol_o = (2 * eps / (1 - eps))[:, None] * vmax + 2.0 ** -9 * np.abs(want_o[i]) + 1e-30
            err_o = np.abs(got_o[t] - want_o[i])
            bad = err_o > tol_o
            assert not bad.any(), (f"request {b} token {t}: {int(bad.sum())} outputs beyond the bound; worst "
                                   f"{float((err_o / tol_o).max()):.3f} x bound")
            tol_l = eps + e_s + 2.0 ** -22 * np.abs(want_lse[i])
            assert np.all(np.abs(got_lse[t] - want_lse[i]) <= tol_l), f"request {b} token {t}: lse"


def run_prefill(kvq, oracle_mod, w, fmt="nvfp4", cache=None, threads=1, requests=None):
    if cache is None:
        cache = host_cache(oracle_mod, w.fill, threads, fmt)
    dcache = torch.from_numpy(cache).to(DEV)
    T, H = w.q.shape[0], w.q.shape[1]
    out = torch.full((T, H, 512), -7.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.full((T, H), -7.0, dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    getattr(kvq, PREFILL_FORMATS[fmt][1])(w.q.to(DEV), w.query_start.to(DEV), w.context_lens.to(DEV),
                                           w.block_table.to(DEV), dcache, w.softmax_scale, w.max_query_len,
                                           out=out, lse=lse, status=status)
    torch.cuda.synchronize()
    check_prefill(oracle_mod, cache, w, out, lse, threads, requests)
    return int(status.item()), out, lse


PREFILL_CASES = [
    # one query token per row block; ragged contexts across 64-position blocks
    ("H128 ragged", dict(context_lens=[100, 64, 257], query_lens=[2, 1, 3], num_heads=128, num_blocks=16,
                         block_size=64, seed=501)),
    # 8 query tokens share every decoded tile; 20 tokens -> 3 row blocks, the last one partial
    ("H16 packed", dict(context_lens=[300, 70], query_lens=[9, 20], num_heads=16, num_blocks=16,
                        block_size=64, seed=502)),
    # 128 / 20 is not whole: a row block holds parts of tokens; an empty context; block size 16
    ("H20 straddling, empty context", dict(context_lens=[130, 0, 65], query_lens=[13, 2, 7], num_heads=20,
                                           num_blocks=24, block_size=16, seed=503)),
    # one head, 200 query tokens: two row blocks of one request
    ("H1 200 tokens", dict(context_lens=[33], query_lens=[200], num_heads=1, num_blocks=4, block_size=16,
                           seed=504)),
    # a request with no query tokens between two that have some
    ("no query tokens", dict(context_lens=[80, 90, 70], query_lens=[1, 0, 2], num_heads=64, num_blocks=8,
                             block_size=64, seed=505)),
]


@pytest.mark.parametrize("fmt", sorted(PREFILL_FORMATS))
@pytest.mark.parametrize("name,kw", PREFILL_CASES, ids=[c[0] for c in PREFILL_CASES])
def test_prefill_parity(kvq, oracle_mod, name, kw, fmt):
    w = wl.make_prefill(name, **kw)
    status, _, _ = run_prefill(kvq, oracle_mod, w, fmt)
    assert status == 0


@pytest.mark.parametrize("fmt", sorted(PREFILL_FORMATS))
def test_prefill_4k_contexts(kvq, oracle_mod, threads, fmt):
    """Contexts of 4096 and 4500 positions (64 and 71 tiles), 128 heads."""
    w = wl.make_prefill("4k contexts", [4096, 4500], [2, 1], 128, 160, 64, 506)
    status, _, _ = run_prefill(kvq, oracle_mod, w, fmt, threads=threads)
    assert status == 0


@pytest.mark.parametrize("fmt", sorted(PREFILL_FORMATS))
def test_prefill_bad_blocks_and_requests(kvq, oracle_mod, fmt):
    """A block id out of range (its positions skipped, KVQ_STATUS_BAD_INDEX),
    a context longer than the table (the rest skipped), and a request whose
    query range runs past num_tokens (skipped whole, KVQ_STATUS_BAD_BATCH,
    its rows untouched)."""
    w = wl.make_prefill("bad", [150, 70, 60], [2, 2, 1], 32, 12, 64, 507)
    table = wl.host(w.block_table).copy()
    table[0, 1] = 1 << 20                            # positions 64..127 of request 0
    w.block_table = torch.from_numpy(table)
    ctx = wl.host(w.context_lens).copy()
    ctx[1] = 200                                     # request 1 owns 2 blocks: positions 128.. skipped
    w.context_lens = torch.from_numpy(ctx)
    qs = wl.host(w.query_start).copy()
    good_qs = qs.copy()
    qs[3] = qs[2] + 5                                # request 2 claims 5 tokens, only 1 exists
    w.query_start = torch.from_numpy(qs)
    w.max_query_len = 5
    cache = host_cache(oracle_mod, w.fill, fmt=fmt)
    dcache = torch.from_numpy(cache).to(DEV)
    T, H = w.q.shape[0], w.q.shape[1]
    out = torch.full((T, H, 512), -7.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.full((T, H), -7.0, dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    getattr(kvq, PREFILL_FORMATS[fmt][1])(w.q.to(DEV), w.query_start.to(DEV), w.context_lens.to(DEV),
                                           w.block_table.to(DEV), dcache, w.softmax_scale, w.max_query_len,
                                           out=out, lse=lse, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == kvq.STATUS_BAD_INDEX | kvq.STATUS_BAD_BATCH
    assert torch.all(out[good_qs[2]:] == -7.0) and torch.all(lse[good_qs[2]:] == -7.0)
    w.query_start = torch.from_numpy(good_qs)
    check_prefill(oracle_mod, cache, w, out, lse, requests=[0, 1])


@pytest.mark.parametrize("fmt", sorted(PREFILL_FORMATS))
def test_prefill_matches_sparse_form(kvq, oracle_mod, fmt):
    """The dense prefill of a request equals the sparse attention of its
    tokens over the slot list of its whole context (the same arithmetic and
    tile order), bit for bit."""
    w = wl.make_prefill("vs sparse", [190, 77], [3, 2], 128, 16, 64, 508)
    cache = host_cache(oracle_mod, w.fill, fmt=fmt)
    dcache = torch.from_numpy(cache).to(DEV)
    q = w.q.to(DEV)
    out, lse = getattr(kvq, PREFILL_FORMATS[fmt][1])(q, w.query_start.to(DEV), w.context_lens.to(DEV),
                                                      w.block_table.to(DEV), dcache, w.softmax_scale,
                                                      w.max_query_len)
    qs, ctx, table = wl.host(w.query_start), wl.host(w.context_lens), wl.host(w.block_table)
    idx = np.full((w.num_tokens, int(ctx.max())), -1, np.int32)
    for b in range(2):
        for t in range(qs[b], qs[b + 1]):
            idx[t, :ctx[b]] = [table[b, p // 64] * 64 + p % 64 for p in range(ctx[b])]
    out2, lse2 = getattr(kvq, FORMATS[fmt][4])(q, torch.from_numpy(idx).to(DEV), dcache, w.softmax_scale)
    torch.cuda.synchronize()
    # equal wherever the token's own list covers the same tiles: all of
    # request 0's tokens (the longest context); request 1's lists are padded
    # with unused entries to the longest context, which adds only masked tiles
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))


@pytest.mark.parametrize("fmt", sorted(PREFILL_FORMATS))
def test_prefill_full_size_sampled(kvq, oracle_mod, threads, fmt):
    """The bench's prefill workload (every request of the prefill gather -- or
    of the fp8 gather -- attends with 16 new tokens x 128 heads to its whole
    context through the gather's block table) in one launch; the first two
    tokens of the request with the shortest and of one with a middle-sized
    context are checked against the oracle."""
    if fmt == "nvfp4":
        gather = wl.prefill_gather(DEV)
    else:
        gather = wl.fp8_gather(DEV)
    w = wl.prefill_attention(gather, DEV)
    cache_host = host_cache(oracle_mod, gather.fill, threads, fmt)
    cache = torch.from_numpy(cache_host).to(DEV)
    del gather
    out, lse = getattr(kvq, PREFILL_FORMATS[fmt][1])(w.q, w.query_start, w.context_lens, w.block_table, cache,
                                                      w.softmax_scale, w.max_query_len)
    torch.cuda.synchronize()
    ctx = wl.host(w.context_lens)
    order = np.argsort(ctx)
    picks = [int(order[0]), int(order[len(order) // 2])]
    # the sampled requests cut down to their first two query tokens
    qs = wl.host(w.query_start)
    keep = torch.from_numpy(np.concatenate([np.arange(qs[b], qs[b] + 2) for b in picks])).to(DEV)
    sub = wl.PrefillWorkload("sampled", None, w.q[keep].cpu(), torch.tensor([0, 2, 4], dtype=torch.int32),
                             torch.from_numpy(ctx[picks].astype(np.int32)),
                             torch.from_numpy(wl.host(w.block_table)[picks]), w.softmax_scale, 2)
    check_prefill(oracle_mod, cache_host, sub, out[keep].cpu(), lse[keep].cpu(), threads)


@pytest.mark.parametrize("layout", ["rows in wider buffers", "heads of a wider tensor"])
def test_query_row_layouts(kvq, oracle_mod, layout):
    """Query rows that are not a packed [T, H, 576] tensor: each row inside a
    640-value buffer (token rows still packed: q_stride_t = H q_stride_h), or
    the first H heads of a tensor with H + 3 heads (token rows not packed).
    The sparse form reads both through its query tensor map; the dense form
    reads the first through its tensor map and copies the second row by row
    itself."""
    T, H = 5, 20

    def place(q):
        q = q.to(DEV)
        if layout == "rows in wider buffers":
            big = torch.zeros((q.shape[0], H, 640), dtype=torch.bfloat16, device=DEV)
            big[:, :, 32:608] = q
            return big[:, :, 32:608]
        big = torch.zeros((q.shape[0], H + 3, 576), dtype=torch.bfloat16, device=DEV)
        big[:, :H] = q
        return big[:, :H]

    w = wl.make_attention("layout sparse", T, H, 128, 8, 64, 521, p_unused=0.1)
    cache = host_cache(oracle_mod, w.fill)
    dcache = torch.from_numpy(cache).to(DEV)
    out, lse = kvq.kvq_sparse_mla_attention_nvfp4_ds_mla(place(w.q), w.indices.to(DEV), dcache, w.softmax_scale)
    torch.cuda.synchronize()
    check(oracle_mod, cache, w.q, wl.host(w.indices), w.softmax_scale, out, lse)

    p = wl.make_prefill("layout dense", [150, 90], [3, 4], H, 8, 64, 522)
    pcache = host_cache(oracle_mod, p.fill)
    out, lse = kvq.kvq_prefill_mla_attention_nvfp4_ds_mla(place(p.q), p.query_start.to(DEV), p.context_lens.to(DEV),
                                                          p.block_table.to(DEV), torch.from_numpy(pcache).to(DEV),
                                                          p.softmax_scale, p.max_query_len)
    torch.cuda.synchronize()
    check_prefill(oracle_mod, pcache, p, out, lse)


# ---------------------------------------------------------------------------
# split-key decode: ranges of a token's keys combined by a second launch
# ---------------------------------------------------------------------------

SPLIT_CASES = [
    # one token, 128 heads, top-2048 in 8 ranges of 4 tiles
    ("1 token top2048 x8", dict(num_tokens=1, num_heads=128, topk=2048, num_blocks=64, block_size=64, seed=531,
                                p_unused=0.1), 8),
    # a ragged list (not whole tiles) in 5 ranges of 2 tiles, the last one partial
    ("3 tokens top300 x5", dict(num_tokens=3, num_heads=64, topk=300, num_blocks=16, block_size=64, seed=532,
                                p_unused=0.2), 5),
    # more ranges than tiles: ranges 2 and 3 are empty
    ("2 tokens top100 x4", dict(num_tokens=2, num_heads=16, topk=100, num_blocks=8, block_size=64, seed=533), 4),
    # the 32-range maximum over a 33-tile list; one head
    ("4 tokens top2100 x32 H1", dict(num_tokens=4, num_heads=1, topk=2100, num_blocks=64, block_size=64,
                                     seed=534, p_unused=0.3), 32),
]


@pytest.mark.parametrize("fmt", sorted(FORMATS))
@pytest.mark.parametrize("name,kw,splits", SPLIT_CASES, ids=[c[0] for c in SPLIT_CASES])
def test_split_parity(kvq, oracle_mod, name, kw, splits, fmt):
    w = wl.make_attention(name, **kw)
    cache = host_cache(oracle_mod, w.fill, fmt=fmt)
    dcache = torch.from_numpy(cache).to(DEV)
    T, H = w.q.shape[0], w.q.shape[1]
    out = torch.full((T, H, 512), -7.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.full((T, H), -7.0, dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    fn = getattr(kvq, FORMATS[fmt][4].replace("sparse_mla_attention", "sparse_mla_attention_split"))
    fn(w.q.to(DEV), w.indices.to(DEV), dcache, w.softmax_scale, num_splits=splits, out=out, lse=lse, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check(oracle_mod, cache, w.q, wl.host(w.indices), w.softmax_scale, out, lse)


def test_split_ranges_without_valid_keys(kvq, oracle_mod):
    """Token 0: its second range (keys 64-127) all unused, weight 0; token 1:
    no valid key at all (out = 0, lse = -inf, as unsplit); a bad slot in
    token 2 is skipped and reported."""
    w = wl.make_attention("split holes", 3, 32, 256, 8, 64, 535)
    idx = wl.host(w.indices).copy()
    idx[0, 64:128] = -1
    idx[1, :] = -1
    idx[2, 10] = 8 * 64 + 3                           # past the cache
    w.indices = torch.from_numpy(idx)
    cache = host_cache(oracle_mod, w.fill)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = kvq.kvq_sparse_mla_attention_split_nvfp4_ds_mla(w.q.to(DEV), w.indices.to(DEV),
                                                               torch.from_numpy(cache).to(DEV), w.softmax_scale,
                                                               num_splits=4, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == kvq.STATUS_BAD_INDEX
    idx[2, 10] = -1                                   # the oracle skips it the same way
    check(oracle_mod, cache, w.q, idx, w.softmax_scale, out, lse)


def test_split_small_batch_full_cache(kvq, oracle_mod, threads):
    """The small-batch case the split serves: 8 decode tokens x 128 heads,
    top-2048 over the 65536 x 64 cache, ranges from default_num_splits, the
    workspace reused by a second call; every token against the oracle."""
    fill = wl.make_fill("split fill", 65536, 64, 1006, DEV, rng="device")
    cache_host = host_cache(oracle_mod, fill, threads)
    cache = torch.from_numpy(cache_host).to(DEV)
    w = wl.make_attention("split decode", 8, 128, 2048, 65536, 64, 536, DEV, p_unused=0.1, fill=fill,
                          rng="device")
    del fill
    splits = kvq.default_num_splits(8, 2048)
    assert splits > 1
    ws = torch.empty(kvq.kvq_sparse_mla_attention_split_workspace_bytes(8, 128, splits), dtype=torch.uint8,
                     device=DEV)
    for _ in range(2):
        out, lse = kvq.kvq_sparse_mla_attention_split_nvfp4_ds_mla(w.q, w.indices, cache, w.softmax_scale,
                                                                   num_splits=splits, workspace=ws)
        torch.cuda.synchronize()
        check(oracle_mod, cache_host, w.q, wl.host(w.indices), w.softmax_scale, out, lse, threads)


def run_prefill_split(kvq, oracle_mod, w, fmt, num_splits, max_context_len=None, requests=None):
    cache = host_cache(oracle_mod, w.fill, fmt=fmt)
    dcache = torch.from_numpy(cache).to(DEV)
    T, H = w.q.shape[0], w.q.shape[1]
    out = torch.full((T, H, 512), -7.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.full((T, H), -7.0, dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    fn = getattr(kvq, PREFILL_FORMATS[fmt][1].replace("prefill_mla_attention", "prefill_mla_attention_split"))
    fn(w.q.to(DEV), w.query_start.to(DEV), w.context_lens.to(DEV), w.block_table.to(DEV), dcache, w.softmax_scale,
       w.max_query_len, max_context_len=max_context_len, num_splits=num_splits, out=out, lse=lse, status=status)
    torch.cuda.synchronize()
    check_prefill(oracle_mod, cache, w, out, lse, requests=requests)
    return int(status.item()), out, lse


@pytest.mark.parametrize("fmt", sorted(PREFILL_FORMATS))
def test_prefill_split_long_context(kvq, oracle_mod, fmt):
    """One request, 3 query tokens x 128 heads over 4500 positions (71
    tiles) in 8 ranges of 9 tiles, the last one partial."""
    w = wl.make_prefill("split long", [4500], [3], 128, 80, 64, 541)
    status, _, _ = run_prefill_split(kvq, oracle_mod, w, fmt, 8)
    assert status == 0


def test_prefill_split_ragged_requests(kvq, oracle_mod):
    """Packed rows of 20 heads, an empty context, a request with no query
    tokens; max_context_len below the longest context (its last range takes
    the rest); 5 ranges."""
    w = wl.make_prefill("split ragged", [700, 0, 90, 1300], [5, 3, 0, 7], 20, 160, 16, 542)
    status, _, _ = run_prefill_split(kvq, oracle_mod, w, "nvfp4", 5, max_context_len=600)
    assert status == 0


def test_prefill_split_untouched_rows(kvq, oracle_mod):
    """Query tokens of no request (before the first one) and of a skipped
    request (its range past num_tokens) keep their outputs; a bad block is
    skipped and reported."""
    w = wl.make_prefill("split holes", [200, 150], [2, 2], 32, 12, 64, 543)
    qs = wl.host(w.query_start).copy()
    table = wl.host(w.block_table).copy()
    table[0, 1] = 1 << 20                            # positions 64..127 of request 0
    w.block_table = torch.from_numpy(table)
    # tokens 0, 1 belong to no request; request 0 = tokens 2-3, request 1 claims 2-7 (only 2-5 exist)
    T = w.num_tokens + 2
    q = torch.zeros((T, 32, 576), dtype=torch.bfloat16)
    q[2:] = w.q
    w.q = q
    w.query_start = torch.from_numpy((qs + 2).astype(np.int32))
    w.query_start[2] = T + 2
    w.max_query_len = 6
    cache = host_cache(oracle_mod, w.fill)
    out = torch.full((T, 32, 512), -7.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.full((T, 32), -7.0, dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvq.kvq_prefill_mla_attention_split_nvfp4_ds_mla(w.q.to(DEV), w.query_start.to(DEV), w.context_lens.to(DEV),
                                                     w.block_table.to(DEV), torch.from_numpy(cache).to(DEV),
                                                     w.softmax_scale, w.max_query_len, num_splits=3, out=out,
                                                     lse=lse, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == kvq.STATUS_BAD_INDEX | kvq.STATUS_BAD_BATCH
    untouched = [0, 1] + list(range(4, T))
    assert torch.all(out[untouched] == -7.0) and torch.all(lse[untouched] == -7.0)
    check_prefill(oracle_mod, cache, w, out, lse, requests=[0])


@pytest.mark.parametrize("fmt", sorted(PREFILL_FORMATS))
def test_prefill_split_full_size_sampled(kvq, oracle_mod, threads, fmt):
    """Two requests of the bench's prefill gather (contexts of the 65536 x 64
    cache, or of the fp8 cache) with 16 query tokens x 128 heads each, split
    with the default range count; the first two tokens of each against the
    oracle."""
    gather = wl.prefill_gather(DEV) if fmt == "nvfp4" else wl.fp8_gather(DEV)
    full = wl.prefill_attention(gather, DEV)
    cache_host = host_cache(oracle_mod, gather.fill, threads, fmt)
    cache = torch.from_numpy(cache_host).to(DEV)
    del gather
    picks = [0, 1]
    qs = wl.host(full.query_start)
    rows = torch.from_numpy(np.concatenate([np.arange(qs[b], qs[b + 1]) for b in picks])).to(DEV)
    sub = wl.PrefillWorkload("split sampled", None, full.q[rows], torch.tensor([0, 16, 32], dtype=torch.int32),
                             full.context_lens[picks].cpu(), full.block_table[picks].cpu(), full.softmax_scale, 16)
    fn = getattr(kvq, PREFILL_FORMATS[fmt][1].replace("prefill_mla_attention", "prefill_mla_attention_split"))
    out, lse = fn(sub.q, sub.query_start.to(DEV), sub.context_lens.to(DEV), sub.block_table.to(DEV), cache,
                  sub.softmax_scale, 16)
    torch.cuda.synchronize()
    keep = torch.tensor([0, 1, 16, 17])
    check_sub = wl.PrefillWorkload("split sampled rows", None, sub.q[keep.to(DEV)].cpu(),
                                   torch.tensor([0, 2, 4], dtype=torch.int32), sub.context_lens,
                                   sub.block_table, sub.softmax_scale, 2)
    check_prefill(oracle_mod, cache_host, check_sub, out[keep.to(DEV)].cpu(), lse[keep.to(DEV)].cpu(), threads)


# ---------------------------------------------------------------------------
# dense prefill over a gathered bf16 workspace (gather, then attention)
# ---------------------------------------------------------------------------

def gather_workspace(kvq, w, dcache, fmt, pad_rows=0):
    """The gather of every request's context into one packed bf16 workspace:
    returns (workspace [sum(ctx) + pad_rows, 576], workspace_starts int32 [B])."""
    ctx = wl.host(w.context_lens).astype(np.int64)
    starts = np.zeros(len(ctx), np.int32)
    starts[1:] = np.cumsum(ctx)[:-1]
    total = int(ctx.sum())
    ws = torch.zeros((total + pad_rows, 576), dtype=torch.bfloat16, device=DEV)
    if total:
        gather = getattr(kvq, "kvq_gather_upconvert_nvfp4_ds_mla" if fmt == "nvfp4" else
                         "kvq_gather_upconvert_fp8_ds_mla")
        gather(dcache, ws[:total], w.block_table.to(DEV), torch.from_numpy(starts).to(DEV),
               torch.zeros(len(ctx), dtype=torch.int32, device=DEV), batch_size=len(ctx))
    return ws, torch.from_numpy(starts).to(DEV)


@pytest.mark.parametrize("fmt", sorted(PREFILL_FORMATS))
@pytest.mark.parametrize("name,kw", PREFILL_CASES, ids=[c[0] for c in PREFILL_CASES])
def test_workspace_prefill_equals_fused(kvq, oracle_mod, name, kw, fmt):
    """Gather + attention over the workspace gives, bit for bit, what the
    fused prefill reads straight from the cache; both against the oracle."""
    w = wl.make_prefill(name, **kw)
    cache = host_cache(oracle_mod, w.fill, fmt=fmt)
    dcache = torch.from_numpy(cache).to(DEV)
    q = w.q.to(DEV)
    ws, starts = gather_workspace(kvq, w, dcache, fmt)
    out, lse = kvq.kvq_prefill_mla_attention_workspace(q, w.query_start.to(DEV), w.context_lens.to(DEV), starts, ws,
                                                       w.softmax_scale, w.max_query_len)
    ref_out, ref_lse = getattr(kvq, PREFILL_FORMATS[fmt][1])(q, w.query_start.to(DEV), w.context_lens.to(DEV),
                                                              w.block_table.to(DEV), dcache, w.softmax_scale,
                                                              w.max_query_len)
    torch.cuda.synchronize()
    qs = wl.host(w.query_start)
    rows = slice(int(qs[0]), int(qs[-1]))                 # tokens of some request
    assert torch.equal(out[rows].view(torch.int16), ref_out[rows].view(torch.int16))
    assert torch.equal(lse[rows].view(torch.int32), ref_lse[rows].view(torch.int32))
    check_prefill(oracle_mod, cache, w, out, lse)


def test_workspace_prefill_4k_and_padding(kvq, oracle_mod, threads):
    """Contexts of 4096 and 4500 positions (the last tile of the second one
    partial), the workspace longer than the contexts (zeroed rows past them)."""
    w = wl.make_prefill("ws 4k", [4096, 4500], [2, 1], 128, 160, 64, 561)
    cache = host_cache(oracle_mod, w.fill, threads)
    ws, starts = gather_workspace(kvq, w, torch.from_numpy(cache).to(DEV), "nvfp4", pad_rows=100)
    out, lse = kvq.kvq_prefill_mla_attention_workspace(w.q.to(DEV), w.query_start.to(DEV), w.context_lens.to(DEV),
                                                       starts, ws, w.softmax_scale, w.max_query_len)
    torch.cuda.synchronize()
    check_prefill(oracle_mod, cache, w, out, lse, threads)


def test_workspace_prefill_bad_ranges(kvq, oracle_mod):
    """A request whose context runs past the workspace and one that starts
    before it are skipped (KVQ_STATUS_BAD_BATCH, rows untouched); the third
    is computed."""
    w = wl.make_prefill("ws bad", [100, 90, 80], [2, 1, 2], 16, 12, 64, 562)
    cache = host_cache(oracle_mod, w.fill)
    ws, starts = gather_workspace(kvq, w, torch.from_numpy(cache).to(DEV), "nvfp4")
    bad = starts.clone()
    bad[0] = int(ws.shape[0]) - 50                    # 100 positions from 50 rows before the end
    bad[1] = -1
    T = w.num_tokens
    out = torch.full((T, 16, 512), -7.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.full((T, 16), -7.0, dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvq.kvq_prefill_mla_attention_workspace(w.q.to(DEV), w.query_start.to(DEV), w.context_lens.to(DEV), bad, ws,
                                            w.softmax_scale, w.max_query_len, out=out, lse=lse, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == kvq.STATUS_BAD_BATCH
    assert torch.all(out[:3] == -7.0) and torch.all(lse[:3] == -7.0)
    check_prefill(oracle_mod, cache, w, out, lse, requests=[2])


@pytest.mark.parametrize("fmt", sorted(PREFILL_FORMATS))
def test_workspace_prefill_full_size_equals_fused(kvq, oracle_mod, threads, fmt):
    """The bench's prefill workloads (32 requests over 7k-34k positions of the
    nvfp4 cache, 16 over the fp8 cache; 16 query tokens x 128 heads each):
    gather + workspace attention equal to the fused prefill bit for bit."""
    gather = wl.prefill_gather(DEV) if fmt == "nvfp4" else wl.fp8_gather(DEV)
    w = wl.prefill_attention(gather, DEV)
    cache = torch.from_numpy(host_cache(oracle_mod, gather.fill, threads, fmt)).to(DEV)
    del gather
    ws, starts = gather_workspace(kvq, w, cache, fmt)
    out, lse = kvq.kvq_prefill_mla_attention_workspace(w.q, w.query_start, w.context_lens, starts, ws,
                                                       w.softmax_scale, w.max_query_len)
    ref_out, ref_lse = getattr(kvq, PREFILL_FORMATS[fmt][1])(w.q, w.query_start, w.context_lens, w.block_table,
                                                              cache, w.softmax_scale, w.max_query_len)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))


def test_trailing_unused_entries(kvq, oracle_mod):
    """Lists that end in unused entries (a context shorter than the list):
    the tiles past the last valid key are skipped.  Token 0 keeps 348 of 2048
    entries and has an out-of-range slot among its unused tail (still
    reported), token 1 keeps 300, token 2 none.  The result equals, bit for
    bit, the one over the lists cut after entry 348, and the oracle's."""
    w = wl.make_attention("trailing", 3, 128, 2048, 64, 64, 571, p_unused=0.1)
    idx = wl.host(w.indices).copy()
    idx[:, 348:] = -1
    idx[1, 300:] = -1
    idx[2, :] = -1
    idx[0, 2000] = 64 * 64 + 5                        # past the cache
    cache = host_cache(oracle_mod, w.fill)
    dcache = torch.from_numpy(cache).to(DEV)
    q = w.q.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = kvq.kvq_sparse_mla_attention_nvfp4_ds_mla(q, torch.from_numpy(idx).to(DEV), dcache, w.softmax_scale,
                                                         status=status)
    cut = np.ascontiguousarray(idx[:, :348])
    out2, lse2 = kvq.kvq_sparse_mla_attention_nvfp4_ds_mla(q, torch.from_numpy(cut).to(DEV), dcache, w.softmax_scale)
    torch.cuda.synchronize()
    assert int(status.item()) == kvq.STATUS_BAD_INDEX
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))
    idx[0, 2000] = -1
    check(oracle_mod, cache, w.q, idx, w.softmax_scale, out, lse)


def test_split_decode_on_a_side_stream_without_lse(kvq, oracle_mod):
    """The split decode's three launches (range marks, partial rows, combine)
    all go to the caller's stream: run on a side stream, no lse output,
    read after that stream alone is synchronised."""
    w = wl.make_attention("split side stream", 3, 64, 512, 16, 64, 581, p_unused=0.1)
    cache = host_cache(oracle_mod, w.fill)
    dcache = torch.from_numpy(cache).to(DEV)
    q, idx = w.q.to(DEV), w.indices.to(DEV)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    out = torch.full((3, 64, 512), -7.0, dtype=torch.bfloat16, device=DEV)
    with torch.cuda.stream(side):
        kvq.kvq_sparse_mla_attention_split_nvfp4_ds_mla(q, idx, dcache, w.softmax_scale, num_splits=4, out=out,
                                                        lse=False, stream=side)
    side.synchronize()
    _, lse_ref, _ = oracle_mod.sparse_mla_attention_nvfp4_ds_mla(wl.bf16_bits(w.q), wl.host(w.indices), cache,
                                                                 w.softmax_scale)
    check(oracle_mod, cache, w.q, wl.host(w.indices), w.softmax_scale, out,
          torch.from_numpy(lse_ref.astype(np.float32)))


def test_workspace_prefill_without_lse(kvq, oracle_mod):
    w = wl.make_prefill("ws no lse", [300, 64], [3, 2], 32, 16, 64, 582)
    cache = host_cache(oracle_mod, w.fill)
    ws, starts = gather_workspace(kvq, w, torch.from_numpy(cache).to(DEV), "nvfp4")
    out, none = kvq.kvq_prefill_mla_attention_workspace(w.q.to(DEV), w.query_start.to(DEV), w.context_lens.to(DEV),
                                                        starts, ws, w.softmax_scale, w.max_query_len, lse=False)
    ref_out, ref_lse = kvq.kvq_prefill_mla_attention_workspace(w.q.to(DEV), w.query_start.to(DEV),
                                                               w.context_lens.to(DEV), starts, ws, w.softmax_scale,
                                                               w.max_query_len)
    torch.cuda.synchronize()
    assert none is None
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    check_prefill(oracle_mod, cache, w, out, ref_lse)
