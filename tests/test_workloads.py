"""The seeded input generators produce what their recipes state (CPU only;
the two multi-GB cache fills are checked through their builders)."""
import numpy as np
import pytest
import torch

import workloads as wl


def test_generators_are_deterministic():
    a, b = wl.smoke_write(), wl.smoke_write()
    assert torch.equal(a.kv_c, b.kv_c) and torch.equal(a.slot_mapping, b.slot_mapping)
    assert a.kv_c.dtype == torch.bfloat16 and a.kv_c.shape == (256, 512) and a.k_pe.shape == (256, 64)


@pytest.mark.parametrize("make,T,slots,pads", [(wl.smoke_write, 256, 512, 16), (wl.decode_write, 8192, 262144, 164)])
def test_write_workloads_slots(make, T, slots, pads):
    w = make()
    s = wl.host(w.slot_mapping)
    assert s.shape == (T,) and w.num_slots == slots
    assert (s < 0).sum() == pads and np.all(s[s < 0] == -1)
    valid = s[s >= 0]
    assert valid.max() < slots and np.unique(valid).size == valid.size


def test_decode_write_outliers():
    x = wl.decode_write().kv_c.float().abs()
    frac = (x > 8).float().mean().item()          # |N(0,1)| > 8 never happens; x50 outliers often do
    assert 0.004 < frac < 0.012


@pytest.mark.parametrize("lens,starts,bs,nb", [([100, 120], [0, 17], 64, 8), ([0, 64, 1, 0, 130], [0, 64, 63, 5, 0], 64, 16),
                                                ([90, 0, 300, 17], [6, 3, 0, 13], 7, 200)])
def test_gather_batch_invariants(lens, starts, bs, nb):
    table, ws, st, T = wl.make_gather_batch(nb, bs, lens, starts, 5)
    assert T == sum(lens) and list(st) == starts
    assert list(ws) == list(np.concatenate([[0], np.cumsum(lens)[:-1]]))
    used = table[table >= 0]
    assert np.unique(used).size == used.size and used.max() < nb          # distinct blocks
    for b, (s, n) in enumerate(zip(starts, lens)):
        need = -(-(s + n) // bs)
        assert np.all(table[b, :need] >= 0) and np.all(table[b, need:] == -1)


def test_smoke_gather_recipe():
    g = wl.smoke_gather()
    assert g.num_out_tokens == 220 and list(wl.host(g.seq_starts)) == [0, 17]
    assert list(wl.host(g.workspace_starts)) == [0, 100]
    f = wl.host(g.fill.slot_mapping)
    assert np.array_equal(np.sort(f), np.arange(512))                  # every slot written once


def test_per_head_recipe():
    w = wl.make_per_head("p", 300, 8, 128, 64, 16, 7, 9)
    assert w.key.shape == (300, 8, 128) and w.value.shape == (300, 8, 128)
    s = wl.host(w.slot_mapping)
    assert (s < 0).sum() == 7 and np.unique(s[s >= 0]).size == 293


def test_nan_free_e4m3_bytes():
    a = np.arange(256, dtype=np.uint8).repeat(3)
    wl.nan_free_e4m3_bytes(a)
    assert not np.any((a & 0x7F) == 0x7F)
