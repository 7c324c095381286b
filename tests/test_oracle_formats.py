"""Pins of the oracle's number-format converters (CPU only).

Each converter is checked against something other than itself: the OCP
golden tables, torch's own float8 / bfloat16 casts (an independent library),
and an exhaustive nearest-value search (tests/independent.py).
"""
import math
import os

import numpy as np
import pytest
import torch

import independent as ind


def test_e2m1_decode_matches_mx_table(oracle_mod):
    for code, val in ind.read_golden("e2m1_values.txt"):
        got = oracle_mod.e2m1_value(int(code, 16))
        want = float(val)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), code


def test_e4m3_decode_matches_torch_for_all_256_codes(oracle_mod):
    want = ind.e4m3_table()
    for c in range(256):
        got = oracle_mod.e4m3_value(c)
        if math.isnan(want[c]):
            assert math.isnan(got), c
        else:
            assert got == want[c] and math.copysign(1, got) == math.copysign(1, want[c]), c


def test_e4m3_decode_landmarks(oracle_mod):
    for code, val in ind.read_golden("e4m3_landmarks.txt"):
        got = oracle_mod.e4m3_value(int(code, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def _strided_bits(stride, offset=0):
    return (np.arange(offset, 1 << 32, stride, dtype=np.uint64)).astype(np.uint32)


def test_e4m3_encode_matches_torch_cast_strided_sweep(oracle_mod):
    """Every 251st float32 bit pattern: inside torch's non-saturating range
    (|f| < 464) the oracle equals torch's RN-even cast; beyond it the oracle
    saturates to +-448 where torch gives NaN."""
    bits = _strided_bits(251, 17)
    f = bits.view(np.float32)
    finite = np.isfinite(f)
    ours = oracle_mod.e4m3_rn_sat(f)
    theirs = ind.torch_e4m3_bits(torch.from_numpy(f.copy())).numpy()
    inr = finite & (np.abs(f) < 464)
    assert inr.sum() > 1_000_000
    np.testing.assert_array_equal(ours[inr], theirs[inr])
    big = ~np.isnan(f) & (np.abs(f) >= 448)
    np.testing.assert_array_equal(ours[big], np.where(np.signbit(f[big]), 0xFE, 0x7E))
    nan = np.isnan(f)
    assert np.all((ours[nan] & 0x7F) == 0x7F)


def test_e4m3_encode_dense_in_interesting_range(oracle_mod):
    """All float32 patterns with exponent in [2^-12, 2^9) every 7th, vs torch."""
    lo = np.float32(2.0 ** -12).view(np.uint32)
    hi = np.float32(2.0 ** 9).view(np.uint32)
    bits = np.arange(int(lo), int(hi), 7, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = np.concatenate([f, -f])
    ours = oracle_mod.e4m3_rn_sat(f)
    m = np.abs(f) < 464
    theirs = ind.torch_e4m3_bits(torch.from_numpy(f[m].copy())).numpy()
    np.testing.assert_array_equal(ours[m], theirs)


def _adjacent_midpoints(mags):
    mids = (mags[:-1] + mags[1:]) / 2.0
    pts = []
    for m in mids:
        m32 = np.float32(m)
        assert float(m32) == m          # midpoints are exact in float32
        pts += [np.nextafter(m32, np.float32(-np.inf)), m32, np.nextafter(m32, np.float32(np.inf))]
    pts += [np.float32(v) for v in mags]
    return np.array(pts, np.float32)


def test_e4m3_encode_bruteforce_at_every_midpoint(oracle_mod):
    mags = ind.e4m3_table()[:127]
    x = _adjacent_midpoints(mags)
    x = np.concatenate([x, -x, np.float32([0.0, -0.0, 1e-45, -1e-45, 2.0 ** -10, 448.0, 464.0, 1e38])])
    np.testing.assert_array_equal(oracle_mod.e4m3_rn_sat(x), ind.e4m3_encode(x))


def test_e4m3_encode_bruteforce_random(oracle_mod):
    g = np.random.Generator(np.random.PCG64(7))
    x = (g.standard_normal(200_000) * np.exp2(g.integers(-14, 10, 200_000))).astype(np.float32)
    np.testing.assert_array_equal(oracle_mod.e4m3_rn_sat(x), ind.e4m3_encode(x))


def test_e2m1_encode_bruteforce_sweep(oracle_mod):
    """Every 13th float32 pattern with |f| in [2^-4, 8), all midpoints +-1 ulp,
    and random magnitudes over a wide range, vs exhaustive search."""
    lo = np.float32(2.0 ** -4).view(np.uint32)
    hi = np.float32(8.0).view(np.uint32)
    f = np.arange(int(lo), int(hi), 13, dtype=np.uint64).astype(np.uint32).view(np.float32)
    mags = ind.e2m1_table()[:8]
    g = np.random.Generator(np.random.PCG64(8))
    r = (g.standard_normal(100_000) * np.exp2(g.integers(-30, 30, 100_000))).astype(np.float32)
    x = np.concatenate([f, -f, _adjacent_midpoints(mags), -_adjacent_midpoints(mags), r,
                        np.float32([0.0, -0.0, 1e-45, -1e-45, 6.0, 7.0, 1e38, -1e38])])
    np.testing.assert_array_equal(oracle_mod.e2m1_rn_sat(x), ind.e2m1_encode(x))


def test_e2m1_rounding_golden(oracle_mod):
    for val, code in ind.read_golden("e2m1_rounding.txt"):
        assert oracle_mod.e2m1_rn_sat(np.float32([float(val)]))[0] == int(code, 16), val


def test_encoders_monotone_and_sign_symmetric(oracle_mod):
    bits = _strided_bits(4099, 3)
    f = bits.view(np.float32)
    f = np.sort(np.abs(f[np.isfinite(f)]))
    for enc, table in ((oracle_mod.e4m3_rn_sat, ind.e4m3_table()), (oracle_mod.e2m1_rn_sat, None)):
        c = enc(f)
        vals = (ind.e4m3_table() if table is not None else ind.e2m1_table())[c]
        assert np.all(np.diff(vals) >= 0)
        neg = enc(-f)
        sign = 0x80 if table is not None else 0x08
        np.testing.assert_array_equal(neg, c | sign)


def test_bf16_rn_matches_torch(oracle_mod):
    g = np.random.Generator(np.random.PCG64(9))
    bits = g.integers(0, 1 << 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    # ties (low half exactly 0x8000) and near-overflow patterns
    ties = (g.integers(0, 1 << 16, size=20_000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    edge = np.array([0x7F7F8000, 0x7F7FFFFF, 0x7F7F7FFF, 0xFF7F8000, 0x00008000, 0x80018000,
                     0x00000001, 0x3F808000, 0x3F818000], np.uint32)
    bits = np.concatenate([bits, ties, edge])
    f = bits.view(np.float32)
    f = f[~np.isnan(f)]
    np.testing.assert_array_equal(oracle_mod.bf16_rn(f), ind.torch_bf16_bits(torch.from_numpy(f.copy())))


def test_bits_range_helpers_agree_with_array_forms(oracle_mod):
    first, n = 0x3E000000, 100_000
    e4, e2 = oracle_mod.encode_bits_range(first, n, threads=4)
    f = np.arange(first, first + n, dtype=np.uint64).astype(np.uint32).view(np.float32)
    np.testing.assert_array_equal(e4, oracle_mod.e4m3_rn_sat(f))
    np.testing.assert_array_equal(e2, oracle_mod.e2m1_rn_sat(f))
    np.testing.assert_array_equal(oracle_mod.bf16_rn_bits_range(first, n, threads=3), oracle_mod.bf16_rn(f))


@pytest.mark.skipif(os.environ.get("KVQ_EXHAUSTIVE_CPU") != "1",
                    reason="all 2^32 patterns: set KVQ_EXHAUSTIVE_CPU=1 (about 10 minutes on 8 cores)")
def test_encoders_exhaustive_against_torch_and_bruteforce(oracle_mod):
    """Every float32 bit pattern: e4m3 against torch's cast inside its
    non-saturating range (and +-448 beyond), e2m1 against the exhaustive
    nearest-value search."""
    chunk = 1 << 24
    threads = oracle_mod.default_threads()
    for first in range(0, 1 << 32, chunk):
        e4, e2 = oracle_mod.encode_bits_range(first, chunk, threads=threads)
        f = np.arange(first, first + chunk, dtype=np.uint64).astype(np.uint32).view(np.float32)
        finite = np.isfinite(f)
        inr = finite & (np.abs(f) < 464)
        t4 = ind.torch_e4m3_bits(torch.from_numpy(f[inr].copy())).numpy()
        assert np.array_equal(e4[inr], t4), hex(first)
        big = ~np.isnan(f) & (np.abs(f) >= 448)
        assert np.array_equal(e4[big], np.where(np.signbit(f[big]), 0xFE, 0x7E)), hex(first)
        assert np.array_equal(e2[finite], ind.e2m1_encode(f[finite])), hex(first)
